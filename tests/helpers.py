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


def oracle_forward(li, tokens=None, nthreads=None):
    """Oracle output (bf16 bits) for the sampled tokens of a LayerInputs (any device)."""
    cpu = lambda t: t.detach().cpu()  # noqa: E731
    return oracle.forward(cpu(li.x), cpu(li.w13), cpu(li.s13), cpu(li.gs13), cpu(li.w2),
                          cpu(li.s2), cpu(li.gs2), cpu(li.topk_ids), cpu(li.topk_weights),
                          tokens=tokens, nthreads=nthreads)


def gpu_forward(li, sched, layer=None):
    from quantized_moe_grouped_route_gb300 import NVFP4MoE
    if layer is None:
        layer = NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    out = layer(li.x, li.topk_ids, li.topk_weights, sched=sched)
    torch.cuda.synchronize()
    return out, layer
