"""Shared helpers for the GPU parity tests (inputs, tolerance, oracle calls)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Per-element bound of the layer's floating-point parity: |got - ref| <= REL*|ref| + ABS*rms(ref)
REL_TOL = 2e-2
RMS_TOL = 2e-3


def to_np_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def check_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = ""):
    got = oracle.bf16_bits_to_float(got_bits)
    ref = oracle.bf16_bits_to_float(ref_bits)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first {idx.tolist()}: got {got[bad][:8]} ref {ref[bad][:8]} "
                             f"(rms {rms:.3g})")
    return float((err / np.maximum(bound, 1e-30)).max()) if err.size else 0.0


# Largest share of h values whose bf16 rounding may differ from the oracle's own: a
# flip is legitimate only when the exact SiLU(gate)*up lies within the GPU's fp32
# rounding noise of a bf16 midpoint (expected rate ~1e-3 or less).
MAX_FLIP_RATE = 5e-3


def oracle_forward(li, tokens=None, nthreads=None, h_given=None, swiglu_limit=None):
    """Oracle output (bf16 bits) for the sampled tokens of a LayerInputs (any device);
    with h_given, also the h-decision statistics."""
    cpu = lambda t: t.detach().cpu()  # noqa: E731
    return oracle.forward(cpu(li.x), cpu(li.w13), cpu(li.s13), cpu(li.gs13), cpu(li.w2),
                          cpu(li.s2), cpu(li.gs2), cpu(li.topk_ids), cpu(li.topk_weights),
                          tokens=tokens, nthreads=nthreads, h_given=h_given,
                          swiglu_limit=swiglu_limit)


def gpu_h_rows(ws, li, sched, tokens) -> np.ndarray:
    """The GPU's bf16 h for each (listed token, slot), [n*top_k][I] bits, read from the
    workspace the last forward call used; zero rows for slots without an expert."""
    from quantized_moe_grouped_route_gb300 import qmoe
    c = li.cfg
    M, top_k = li.x.shape[0], li.topk_ids.shape[1]
    v = qmoe.workspace_views(ws, M, c.H, c.I, c.E, top_k, sched)
    pp = v["pair_pos"].cpu().numpy()
    h = v["h"].cpu().view(torch.int16).numpy().astype(np.uint16)
    pairs = np.array([m * top_k + k for m in tokens for k in range(top_k)], np.int64)
    pos = pp[pairs] if pairs.size else np.zeros(0, np.int64)
    out = np.zeros((pairs.size, c.I), np.uint16)
    ok = pos >= 0
    out[ok] = h[pos[ok]]
    return out


def check_layer(li, out, ws, sched, tokens=None, what="", swiglu_limit=None):
    """Parity of one forward call: (1) every GPU h value is one of the two bf16 values
    bracketing the exact SiLU(gate)*up and at most MAX_FLIP_RATE of them differ from
    the oracle's own rounding; (2) the outputs match the oracle fed those h decisions,
    per element within the layer tolerance."""
    M = li.x.shape[0]
    toks = np.arange(M) if tokens is None else np.asarray(tokens)
    hg = gpu_h_rows(ws, li, sched, toks)
    ref, st = oracle_forward(li, tokens=toks, h_given=hg, swiglu_limit=swiglu_limit)
    assert st["outside"] == 0, f"{what}: {st['outside']} h values outside their bf16 bracket"
    assert st["flipped"] <= MAX_FLIP_RATE * max(st["compared"], 1), \
        f"{what}: {st['flipped']} of {st['compared']} h roundings differ"
    got = to_np_bf16_bits(out)[toks]
    ratio = check_close(got, ref, what)
    return {"h_compared": st["compared"], "h_flipped": st["flipped"], "max_ratio": ratio}


def gpu_forward(li, sched, layer=None, swiglu_limit=None):
    from quantized_moe_grouped_route_gb300 import NVFP4MoE
    if layer is None:
        layer = NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    out = layer(li.x, li.topk_ids, li.topk_weights, sched=sched, swiglu_limit=swiglu_limit)
    torch.cuda.synchronize()
    return out, layer
