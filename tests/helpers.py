"""Shared helpers for the GPU parity tests (inputs, tolerance, oracle calls)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Per-element bound of the layer's floating-point parity: |got - ref| <= REL*|ref| + ABS*rms(ref)
REL_TOL = 2e-2
RMS_TOL = 2e-3

# Largest share of h values whose bf16 rounding may differ from the oracle's own.  A
# flip is legitimate only when the exact SiLU(gate)*up lies within the GPU's fp32
# accumulation noise of a bf16 rounding midpoint.  The limit comes from an emulation of
# that accumulation at H = 7168 (tests/test_h_rounding_bound.py): 3.4e-4 of the values
# flip with round-to-nearest additions, 1.4e-3 with truncating ones (the least
# favourable rounding, and the one the GPU's measured rates match: 1.6e-3 on the large
# prefill workload); the limit is about twice the truncating rate.
MAX_FLIP_RATE = 3e-3

# Largest share of compared output elements allowed outside the tolerance against the
# unconditioned oracle; each of them must also be explained by a validated h flip in
# its own token (check_layer).
MAX_EXPLAINED_RATE = 1e-4


def to_np_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def rms_of(ref_bits: np.ndarray) -> float:
    ref = oracle.bf16_bits_to_float(ref_bits)
    return float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0


def out_of_tolerance(got_bits: np.ndarray, ref_bits: np.ndarray, rms: float) -> np.ndarray:
    """Boolean mask of the elements with |got - ref| > REL*|ref| + RMS*rms."""
    got = oracle.bf16_bits_to_float(got_bits)
    ref = oracle.bf16_bits_to_float(ref_bits)
    return ~(np.abs(got - ref) <= REL_TOL * np.abs(ref) + RMS_TOL * rms)


def check_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = ""):
    got = oracle.bf16_bits_to_float(got_bits)
    ref = oracle.bf16_bits_to_float(ref_bits)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = rms_of(ref_bits)
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(got - ref)
    bad = out_of_tolerance(got_bits, ref_bits, rms)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first {idx.tolist()}: got {got[bad][:8]} ref {ref[bad][:8]} "
                             f"(rms {rms:.3g})")
    return float((err / np.maximum(bound, 1e-30)).max()) if err.size else 0.0


def oracle_forward(li, tokens=None, nthreads=None, h_given=None, swiglu_limit=None,
                   return_h=False):
    """Oracle output (bf16 bits) for the sampled tokens of a LayerInputs (any device);
    with h_given or return_h, also the h used and the h-decision statistics."""
    cpu = lambda t: t.detach().cpu()  # noqa: E731
    return oracle.forward(cpu(li.x), cpu(li.w13), cpu(li.s13), cpu(li.gs13), cpu(li.w2),
                          cpu(li.s2), cpu(li.gs2), cpu(li.topk_ids), cpu(li.topk_weights),
                          tokens=tokens, nthreads=nthreads, h_given=h_given,
                          swiglu_limit=swiglu_limit, return_h=return_h)


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
    """Parity of one forward call against the oracle on the listed tokens (all by default).

    1. The GPU output is compared element by element with the unconditioned oracle (its
       own fp64 arithmetic and its own bf16 rounding of h) within the layer tolerance.
    2. The GPU's bf16 h is read back.  Where it differs from the oracle's rounding (a
       "flip"), the value must be a valid rounding: the oracle, handed those values,
       checks each against the bracket of the exact SiLU(gate)*up widened by an fp32
       accumulation error bound.  Flips must stay under MAX_FLIP_RATE of the h values.
    3. An output element outside the tolerance of step 1 is accepted only when (i) its
       token has at least one validated flip, (ii) the element is within the tolerance
       of the oracle fed the GPU's h decisions, and (iii) such elements are at most
       MAX_EXPLAINED_RATE of those compared.
    Returns the counts of each step."""
    M = li.x.shape[0]
    top_k = li.topk_ids.shape[1]
    toks = np.arange(M) if tokens is None else np.asarray(tokens)
    got = to_np_bf16_bits(out)[toks]
    assert np.isfinite(oracle.bf16_bits_to_float(got)).all(), f"{what}: non-finite output"
    ref, info = oracle_forward(li, tokens=toks, swiglu_limit=swiglu_limit, return_h=True)
    hg = gpu_h_rows(ws, li, sched, toks)
    flips = hg != info["h"]                                  # [n*top_k][I]
    ids = li.topk_ids.cpu().numpy()[toks]
    n_h = int(((ids >= 0) & (ids < li.cfg.E)).sum()) * hg.shape[1]
    n_flip = int(flips.sum())
    flip_tok = np.nonzero(flips.reshape(len(toks), -1).any(axis=1))[0]   # indices into toks
    ref_h = ref.copy()
    if flip_tok.size:
        rows = (flip_tok[:, None] * top_k + np.arange(top_k)[None, :]).reshape(-1)
        r2, st = oracle_forward(li, tokens=toks[flip_tok], h_given=hg[rows],
                                swiglu_limit=swiglu_limit)
        assert st["outside"] == 0, f"{what}: {st['outside']} h values outside their bf16 bracket"
        assert st["flipped"] == n_flip
        ref_h[flip_tok] = r2
    assert n_flip <= MAX_FLIP_RATE * max(n_h, 1), f"{what}: {n_flip} of {n_h} h roundings differ"
    rms = rms_of(ref)
    bad = out_of_tolerance(got, ref, rms)
    n_bad = int(bad.sum())
    if n_bad:
        bad_tok = np.unique(np.nonzero(bad)[0])
        unexplained = np.setdiff1d(bad_tok, flip_tok)
        assert unexplained.size == 0, (
            f"{what}: {n_bad} of {bad.size} outputs out of tolerance against the oracle, in "
            f"tokens {toks[unexplained][:8].tolist()} that have no h flip")
        still = bad & out_of_tolerance(got, ref_h, rms)
        assert not still.any(), (
            f"{what}: {int(still.sum())} outputs out of tolerance even against the oracle fed "
            f"the GPU's h decisions")
        assert n_bad <= MAX_EXPLAINED_RATE * bad.size, (
            f"{what}: {n_bad} of {bad.size} outputs outside the tolerance against the oracle "
            f"(each explained by an h flip, but more than {MAX_EXPLAINED_RATE:g} of them)")
    print(f"[parity] {what}: {bad.size} outputs compared, {n_bad} outside the tolerance "
          f"against the unconditioned oracle; {n_h} h values, {n_flip} rounded the other way "
          f"(in {flip_tok.size} of {len(toks)} tokens)")
    return {"compared": int(bad.size), "outside_unconditioned": n_bad, "h_compared": n_h,
            "h_flipped": n_flip, "flip_tokens": int(flip_tok.size)}


def forced_tokens(li, sched, n_random=64, seed=0):
    """Tokens to check on a full-size workload: n_random drawn uniformly, plus tokens with
    a pair at the places a schedule is most likely to go wrong: the last and first pair
    of the heaviest expert's tail tile, pairs of the three lightest touched experts, and
    pairs in the second MMA chain of a tile wider than 256 pairs."""
    from quantized_moe_grouped_route_gb300 import qmoe
    ids = li.topk_ids.cpu().numpy()
    M, k = ids.shape
    E = li.cfg.E
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E)
    # stable rank of each pair among the pairs of its expert
    order = np.argsort(np.where(valid, flat, E), kind="stable")
    rank = np.full(flat.size, -1, np.int64)
    starts = np.concatenate([[0], np.cumsum(counts)])
    for e in np.nonzero(counts)[0]:
        rank[order[starts[e]:starts[e + 1]]] = np.arange(counts[e])
    tile_n = qmoe.qmoe_sched_tile_n(sched, M, k, E)
    pairs = []
    heavy = int(counts.argmax())
    last = int(counts[heavy]) - 1
    tail0 = (last // tile_n) * tile_n
    for r in (last, tail0):
        pairs += np.nonzero((flat == heavy) & (rank == r))[0][:1].tolist()
    touched = np.nonzero(counts)[0]
    for e in touched[np.argsort(counts[touched], kind="stable")][:3]:
        pairs += np.nonzero(flat == e)[0][:2].tolist()
    if tile_n > 256:
        second = np.nonzero(valid & (rank % tile_n >= 256))[0]
        pairs += second[:4].tolist()
    forced = np.unique(np.asarray(pairs, np.int64) // k)
    rng = np.random.default_rng(seed)
    rand = rng.choice(M, size=min(M, n_random), replace=False)
    return np.unique(np.concatenate([[0, M - 1], forced, rand])).astype(np.int64)


def gpu_forward(li, sched, layer=None, swiglu_limit=None):
    from quantized_moe_grouped_route_gb300 import NVFP4MoE
    if layer is None:
        layer = NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    out = layer(li.x, li.topk_ids, li.topk_weights, sched=sched, swiglu_limit=swiglu_limit)
    torch.cuda.synchronize()
    return out, layer
