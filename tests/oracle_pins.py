"""Pins for the CPU oracle: checks that tie it to facts other than itself.

Each ``pin_*`` function takes a loaded oracle library and raises AssertionError on
a mismatch.  ``test_oracle_pins.py`` runs them against the real oracle and, with
mistakes planted in copies of the oracle source, shows that every planted mistake
fails at least one pin.  Expected values come from closed forms, library routines
(torch's float8 / bf16 conversions, Python's ``sorted``), brute force over all
bf16 values, and invariants of the layer; none comes from the oracle itself.
"""

from __future__ import annotations

import math
import random

import numpy as np
import torch

import oracle

# E2M1 magnitudes as the NVFP4 format defines them (sign in bit 3).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]

_ALL_BF16 = None


def all_bf16_values():
    """float64 value of every finite, non-negative bf16 bit pattern (index = bits)."""
    global _ALL_BF16
    if _ALL_BF16 is None:
        bits = torch.arange(0, 0x7F80, dtype=torch.int32).to(torch.int16)
        _ALL_BF16 = bits.view(torch.bfloat16).double().numpy()
    return _ALL_BF16


def brute_bf16(v: float) -> int:
    """bf16 bits of the bf16 value nearest to v (ties: even bit pattern), by search."""
    vals = all_bf16_values()
    a = abs(v)
    if a >= 2.0 ** 128 * (1 - 2.0 ** -9):
        mag = 0x7F80
    else:
        i = int(np.searchsorted(vals, a))
        cands = [j for j in (i - 1, i, i + 1) if 0 <= j < vals.size]
        best = min(cands, key=lambda j: (abs(vals[j] - a), j & 1))
        mag = best
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    return sign | mag


def bits_to_f(bits: int) -> float:
    return float(torch.tensor([bits & 0xFFFF], dtype=torch.int32).to(torch.int16)
                 .view(torch.bfloat16).double()[0])


def silu(g: float) -> float:
    return g / (1.0 + math.exp(-g))


# ---------------------------------------------------------------------------
# format decoders
# ---------------------------------------------------------------------------

def pin_e2m1(lib):
    for c in range(16):
        closed = (-1.0 if c & 8 else 1.0) * (
            (c & 1) * 0.5 if (c >> 1) & 3 == 0 else 2.0 ** (((c >> 1) & 3) - 1) * (1 + 0.5 * (c & 1)))
        want = (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7]
        assert closed == want or (closed == 0 and want == 0)
        got = oracle.dec_e2m1(c, lib)
        assert got == want, (c, got, want)


def pin_e4m3(lib):
    lib_vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double()
    for b in range(256):
        got = oracle.dec_e4m3(b, lib)
        want = float(lib_vals[b])
        if b & 0x7F == 0x7F:
            assert math.isnan(got), b
            continue
        assert got == want, (b, got, want)
    assert oracle.dec_e4m3(0x7E, lib) == 448.0
    assert oracle.dec_e4m3(0x01, lib) == 2.0 ** -9
    assert oracle.dec_e4m3(0x08, lib) == 2.0 ** -6
    assert oracle.dec_e4m3(0x38, lib) == 1.0
    assert oracle.dec_e4m3(0xB8, lib) == -1.0


def pin_bf16_decode(lib):
    vals = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = vals.double().numpy()
    rng = random.Random(5)
    idx = list(range(0, 65536, 7)) + [rng.randrange(65536) for _ in range(2000)]
    for i in idx:
        bits = (i - 32768) & 0xFFFF
        got = oracle.bf16_to_double(bits, lib)
        want = vals[i]
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want, (hex(bits), got, want)


def pin_bf16_round(lib):
    # values exactly representable in fp32: torch's fp32 -> bf16 rounding is a single RNE
    g = torch.Generator().manual_seed(11)
    f = torch.randn(4000, generator=g) * torch.exp2(torch.randint(-140, 120, (4000,), generator=g)
                                                     .float())
    f = torch.cat([f, torch.tensor([0.0, -0.0, 1.0, -3.5, 2.0 ** -130, 3e38, -3.3e38])])
    want = f.to(torch.bfloat16).view(torch.int16).int().numpy() & 0xFFFF
    for v, w in zip(f.double().tolist(), want.tolist()):
        assert oracle.bf16_rne(v, lib) == w, (v, hex(oracle.bf16_rne(v, lib)), hex(w))
    # ties and values only a double can hold (no double rounding through fp32)
    cases = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40,
             -(1.0 + 2.0 ** -8 + 2.0 ** -40), 2.0 ** -134, 1.5 * 2.0 ** -134, 2.0 ** -133,
             (2 - 2.0 ** -8) * 2.0 ** 127, (2 - 2.0 ** -7) * 2.0 ** 127, 6.0e-39, 1e-45]
    for v in cases:
        assert oracle.bf16_rne(v, lib) == brute_bf16(v), (v, hex(oracle.bf16_rne(v, lib)),
                                                          hex(brute_bf16(v)))
    assert oracle.bf16_rne(1.0 + 2.0 ** -8, lib) == 0x3F80
    assert oracle.bf16_rne(1.0 + 3 * 2.0 ** -8, lib) == 0x3F82
    assert oracle.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -40, lib) == 0x3F81


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def _route_brute(ids, E, T):
    P = len(ids)
    valid = [i for i in range(P) if 0 <= ids[i] < E]
    order = sorted(valid, key=lambda i: (ids[i], i))
    offsets = [sum(1 for i in valid if ids[i] < e) for e in range(E + 1)]
    pair_pos = [-1] * P
    for pos, i in enumerate(order):
        pair_pos[i] = pos
    sorted_pair = order + [-1] * (P - len(order))
    tiles = []
    for e in range(E):
        s = offsets[e]
        while s < offsets[e + 1]:
            tiles.append((e, s, min(T, offsets[e + 1] - s)))
            s += T
    return offsets, sorted_pair, pair_pos, tiles


def pin_route(lib):
    rng = np.random.default_rng(3)
    cases = []
    for (P, E, T) in [(8, 8, 16), (128, 256, 16), (300, 7, 16), (1000, 3, 128), (64, 1, 16),
                      (0, 4, 16), (50, 5, 1), (257, 2, 256)]:
        ids = rng.integers(-1, E, size=P).astype(np.int32)
        cases.append((ids, E, T))
    cases.append((np.full(40, 2, np.int32), 4, 16))     # all pairs on one expert
    cases.append((np.full(17, -1, np.int32), 4, 16))    # nothing routed
    for ids, E, T in cases:
        off, sp, pp, tiles, rc = oracle.route(ids, E, T, lib=lib)
        b_off, b_sp, b_pp, b_tiles = _route_brute(ids.tolist(), E, T)
        assert rc == 0
        assert off.tolist() == b_off
        assert sp.tolist() == b_sp
        assert pp.tolist() == b_pp
        assert [tuple(t) for t in tiles.tolist()] == b_tiles
    # ids >= E are skipped like -1 and reported
    ids = np.array([0, 5, 1, -1, 9, 1], np.int32)
    off, sp, pp, tiles, rc = oracle.route(ids, 3, 2, lib=lib)
    assert rc == oracle.QO_WARN_BAD_ID
    assert off.tolist() == [0, 1, 3, 3]
    assert sp.tolist() == [0, 2, 5, -1, -1, -1]
    assert pp.tolist() == [0, -1, 1, -1, -1, 2]
    assert [tuple(t) for t in tiles.tolist()] == [(0, 0, 1), (1, 1, 2)]


# ---------------------------------------------------------------------------
# the layer: closed forms on hand-built weights
# ---------------------------------------------------------------------------

def _zeros(M, H, I, E, top_k):
    return dict(
        x=np.zeros((M, H), np.uint16),
        w13=np.zeros((E, 2 * I, H // 2), np.uint8), s13=np.zeros((E, 2 * I, H // 16), np.uint8),
        gs13=np.ones(E, np.float32),
        w2=np.zeros((E, H, I // 2), np.uint8), s2=np.zeros((E, H, I // 16), np.uint8),
        gs2=np.ones(E, np.float32),
        topk_ids=np.zeros((M, top_k), np.int32), topk_weights=np.ones((M, top_k), np.float32))


def _set_code(w, s, e, n, k, code, scale_byte):
    byte = int(w[e, n, k // 2])
    if k % 2 == 0:
        byte = (byte & 0xF0) | code
    else:
        byte = (byte & 0x0F) | (code << 4)
    w[e, n, k // 2] = byte
    s[e, n, k // 16] = scale_byte


def _rand_bf16(rng, shape, scale=1.0):
    v = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
    return v.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def _run(lib, t, **kw):
    return oracle.forward(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"], t["s2"], t["gs2"],
                          t["topk_ids"], t["topk_weights"], lib=lib, nthreads=2, **kw)


def pin_zero_weights(lib):
    rng = np.random.default_rng(0)
    t = _zeros(3, 64, 32, 2, 2)
    t["x"] = _rand_bf16(rng, (3, 64))
    t["topk_ids"] = np.array([[0, 1], [1, 0], [0, -1]], np.int32)
    out = _run(lib, t)
    assert (out & 0x7FFF == 0).all()


def _single_nibble_layer():
    rng = np.random.default_rng(1)
    M, H, I, E = 2, 64, 32, 3
    t = _zeros(M, H, I, E, 1)
    t["x"] = _rand_bf16(rng, (M, H))
    e, i0, j0 = 2, 5, 37
    ku, kg = 19, 42            # odd k -> high nibble, even k -> low nibble
    _set_code(t["w13"], t["s13"], e, i0, ku, 0x5, 0x3A)         # +3.0 ; 1.25
    _set_code(t["w13"], t["s13"], e, I + i0, kg, 0xC, 0x41)     # -2.0 ; 2.25
    _set_code(t["w2"], t["s2"], e, j0, i0, 0x7, 0x2C)           # +6.0 ; 0.375
    t["gs13"][:] = [7.0, 7.0, 0.75]
    t["gs2"][:] = [5.0, 5.0, 1.5]
    t["topk_ids"][:] = [[e], [e]]
    t["topk_weights"][:] = [[0.625], [-1.75]]
    geo = dict(M=M, H=H, I=I, i0=i0, j0=j0, ku=ku, kg=kg)
    return t, geo


def _single_nibble_h(t, geo, m):
    xu = bits_to_f(int(t["x"][m, geo["ku"]]))
    xg = bits_to_f(int(t["x"][m, geo["kg"]]))
    up = 0.75 * 3.0 * 1.25 * xu
    gate = 0.75 * -2.0 * 2.25 * xg
    return silu(gate) * up


def pin_single_nibble(lib):
    """One nonzero code per matrix: every factor of the output is known in closed form."""
    t, geo = _single_nibble_layer()
    out = _run(lib, t)
    for m in range(geo["M"]):
        h = bits_to_f(brute_bf16(_single_nibble_h(t, geo, m)))
        y = 1.5 * 6.0 * 0.375 * h
        want = brute_bf16(float(t["topk_weights"][m, 0]) * y)
        for j in range(geo["H"]):
            expect = want if j == geo["j0"] else 0
            mask = 0xFFFF if j == geo["j0"] else 0x7FFF
            assert (int(out[m, j]) & mask) == expect, (m, j, out[m, j], expect)


def _bf16_neighbors(v):
    """(lo, hi) bf16 bit patterns bracketing v, by brute force over all bf16 values."""
    vals = all_bf16_values()
    a = abs(v)
    i = int(np.searchsorted(vals, a, side="right")) - 1   # largest value <= a
    lo_mag, hi_mag = i, (i if vals[i] == a else i + 1)
    sign = 0x8000 if v < 0 else 0
    if v < 0:
        lo_mag, hi_mag = hi_mag, lo_mag
    return sign | lo_mag, sign | hi_mag


def pin_h_given(lib):
    """h decisions handed to the oracle: checked against the bracket of the exact value
    and used for FC2 at the right index."""
    t = _random_layer(21, M=4, H=64, I=32, E=3, top_k=2)
    t["topk_ids"][1, 1] = -1
    out, f64, info = _run(lib, t, return_f64=True, return_h=True)
    n_valid = int((t["topk_ids"] >= 0).sum())
    out2, f64b, st = _run(lib, t, return_f64=True, h_given=info["h"])
    assert np.array_equal(out, out2) and np.array_equal(f64, f64b)
    assert st["compared"] == n_valid * 32 and st["flipped"] == 0 and st["outside"] == 0
    assert not info["h"][1 * 2 + 1].any()   # slot without an expert: zero row

    t, geo = _single_nibble_layer()
    I, i0, j0 = geo["I"], geo["i0"], geo["j0"]
    for m_try in range(geo["M"]):
        exact = _single_nibble_h(t, geo, m_try)
        lo, hi = _bf16_neighbors(exact)
        rne = brute_bf16(exact)
        other = hi if rne == lo else lo
        hg = np.zeros((geo["M"], I), np.uint16)
        for m in range(geo["M"]):
            hg[m, i0] = brute_bf16(_single_nibble_h(t, geo, m))
        hg[m_try, i0] = other
        o, st = _run(lib, t, h_given=hg)
        assert st["compared"] == geo["M"] * I and st["flipped"] == 1 and st["outside"] == 0
        y = 1.5 * 6.0 * 0.375 * bits_to_f(other)
        assert int(o[m_try, j0]) == brute_bf16(float(t["topk_weights"][m_try, 0]) * y)
        # two steps away from the exact value is not a valid rounding
        far = (other + 1) if (other & 0x8000) == 0 and other == hi else other
        if far == other:
            far = (hi + 1) if (hi & 0x8000) == 0 else (hi - 1)
        hg[m_try, i0] = far
        _, st = _run(lib, t, h_given=hg)
        assert st["outside"] == 1


# ---------------------------------------------------------------------------
# the h-acceptance bound at production size, against emulated fp32 accumulation
# ---------------------------------------------------------------------------

EMU_SLICE = 16    # K per tcgen05 MMA of kind::f16
EMU_STEP = 256    # K per pipeline step of the decode schedule (its MMA warps alternate)


def _round32(v64, truncate):
    """float64 -> float32, to nearest (ties to even) or toward zero."""
    t = v64.astype(np.float32)
    if truncate:
        over = np.abs(t.astype(np.float64)) > np.abs(v64)
        t = np.where(over, np.nextafter(t, np.float32(0)), t)
    return t


def _add32(a, b, truncate):
    # the sum of two float32 values is exact in float64 at the magnitudes met here
    return _round32(a.astype(np.float64) + b.astype(np.float64), truncate)


def emulate_fc1_h(x, w13, gs, chains, truncate):
    """bf16 bits of h = SiLU(gate) * up as the grouped GEMM forms them, emulated:
    x [M][H] bf16 values and w13 [2I][H] exact dequantized weights (float64); products
    exact, each 16-wide K slice sum rounded to fp32 and added to an fp32 accumulator,
    the 256-wide K steps dealt round robin over `chains` accumulators which are added
    in order at the end; every rounding to nearest or toward zero (`truncate`); then
    the global scale, SiLU and the product in fp32 and a round to bf16."""
    M, H = x.shape
    N = w13.shape[0]
    ns = H // EMU_SLICE
    xs = x.reshape(M, ns, EMU_SLICE).transpose(1, 0, 2)
    ws = w13.reshape(N, ns, EMU_SLICE).transpose(1, 2, 0)
    slices = np.matmul(xs, ws)                               # [slice][m][n], fp64
    acc = np.zeros((chains, M, N), np.float32)
    per_step = EMU_STEP // EMU_SLICE
    for s_ in range(ns):
        c = (s_ // per_step) % chains
        acc[c] = _add32(acc[c], _round32(slices[s_], truncate), truncate)
    v = np.zeros((M, N), np.float32)
    for c in range(chains):
        v = _add32(v, acc[c], truncate)
    g = _round32(v.astype(np.float64) * np.float64(np.float32(gs)), False)
    I = N // 2
    up, gate = g[:, :I], g[:, I:]
    with np.errstate(over="ignore"):
        e = np.exp(-gate).astype(np.float32)
    h32 = ((gate / (np.float32(1) + e)).astype(np.float32) * up).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(h32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().astype(np.uint16)


def h_bound_layer(M, I, seed=101, H=7168):
    """One expert, one slot per token: the h-given statistics of each token's h."""
    from qmoe_inputs import LayerConfig, make_inputs
    from oracle import ref_numpy
    li = make_inputs(LayerConfig(f"hbound_m{M}_h{H}_i{I}", M, H, I, 1, 1, seed=seed), "cpu")
    li.topk_weights = torch.ones_like(li.topk_weights)
    x = oracle.bf16_bits_to_float(li.x.view(torch.int16).numpy().astype(np.uint16))
    w13 = ref_numpy.dequant(li.w13[0].numpy(), li.s13[0].numpy())
    return li, x, w13, float(li.gs13[0])


def h_given_stats(lib, li, hg):
    _, st = oracle.forward(li.x, li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2, li.topk_ids,
                           li.topk_weights, h_given=hg, lib=lib)
    return st


def two_steps_away(own, direction):
    """bf16 bits moved `direction` (+2 / -2) steps in magnitude; tiny and huge values kept."""
    mag = own & 0x7FFF
    ok = (mag >= 4) & (mag < 0x7F00)
    far = np.where(ok, own.astype(np.int32) + direction, own.astype(np.int32)).astype(np.uint16)
    return far, int(ok.sum())


def cancelling_layer(M, I, seed=103, H=7168):
    """h_bound_layer whose dot products cancel: the second half of K repeats the first
    half of x with every weight's sign flipped (same scales), and one activation of the
    second half is perturbed, so the exact g is small while the running sums of the
    accumulation are not: the fp32 error then spans many bf16 steps of h."""
    li, x, w13, gs = h_bound_layer(M, I, seed=seed, H=H)
    half = H // 2
    w = li.w13[0].numpy()
    w[:, half // 2:] = w[:, : half // 2] ^ 0x88          # both nibbles' sign bits
    sc = li.s13[0].numpy()
    sc[:, half // 16:] = sc[:, : half // 16]
    xb = li.x.view(torch.int16).numpy()
    xb[:, half:] = xb[:, :half]
    xb[:, H - 1] = np.int16(0x3F80)                       # 1.0
    from oracle import ref_numpy
    x = oracle.bf16_bits_to_float(xb.astype(np.uint16))
    w13 = ref_numpy.dequant(w, sc)
    return li, x, w13, gs


_HB = None
_HC = None


def pin_h_bound_production(lib):
    """At H = 7168 every emulated fp32 accumulation (one or three accumulators, rounding
    to nearest or truncating) is accepted, and values two bf16 steps from the oracle's
    own rounding are rejected except where the exact value's error bound is that wide
    (cancelling dot products: under 2% here)."""
    global _HB
    if _HB is None:
        _HB = h_bound_layer(16, 256)
    li, x, w13, gs = _HB
    for chains, trunc in ((1, True), (3, True), (1, False)):
        st = h_given_stats(lib, li, emulate_fc1_h(x, w13, gs, chains, trunc))
        assert st["compared"] == 16 * 256 and st["outside"] == 0, (chains, trunc, st)
    own = oracle.forward(li.x, li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2, li.topk_ids,
                         li.topk_weights, return_h=True, lib=lib)[1]["h"]
    for d in (2, -2):
        far, moved = two_steps_away(own, d)
        st = h_given_stats(lib, li, far)
        assert moved - st["outside"] <= 0.02 * moved, (d, moved, st)
    # cancelling dot products: the emulated accumulations land several bf16 steps from
    # the exact value, where only the running-sum part of the bound admits them
    global _HC
    if _HC is None:
        _HC = cancelling_layer(16, 128)
    li, x, w13, gs = _HC
    for chains, trunc in ((1, True), (3, True), (1, False)):
        st = h_given_stats(lib, li, emulate_fc1_h(x, w13, gs, chains, trunc))
        assert st["outside"] == 0, (chains, trunc, st)
        if trunc:
            assert st["flipped"] >= st["compared"] // 8, st


def pin_permutation_blocks(lib):
    """Permutation-matrix weights: up[i] = x[sig(i)], gate[i] = 2 x[tau(i)],
    out[j] = h[pi(j)] with h = bf16(silu(gate) * up)."""
    rng = np.random.default_rng(2)
    M, H, I, E = 3, 48, 32, 2
    t = _zeros(M, H, I, E, 2)
    t["x"] = _rand_bf16(rng, (M, H))
    sig = rng.permutation(H)[:I]
    tau = rng.permutation(H)[:I]
    pi = rng.integers(0, I, size=H)
    e = 1
    for i in range(I):
        _set_code(t["w13"], t["s13"], e, i, int(sig[i]), 0x2, 0x40)       # 1.0 * 2.0
        _set_code(t["w13"], t["s13"], e, I + i, int(tau[i]), 0x4, 0x40)   # 2.0 * 2.0
    for j in range(H):
        _set_code(t["w2"], t["s2"], e, j, int(pi[j]), 0xA, 0x30)           # -1.0 * 0.5
    t["gs13"][e] = 0.5
    t["gs2"][e] = -2.0
    t["topk_ids"][:] = [[e, -1], [-1, e], [e, 0]]
    t["topk_weights"][:] = [[1.0, 9.0], [3.0, 1.0], [1.0, 0.0]]
    out = _run(lib, t)
    for m in range(M):
        xm = [bits_to_f(int(b)) for b in t["x"][m]]
        h = [bits_to_f(brute_bf16(silu(2.0 * xm[tau[i]]) * xm[sig[i]])) for i in range(I)]
        for j in range(H):
            assert int(out[m, j]) == brute_bf16(h[pi[j]]), (m, j)


def pin_subnormal_scale(lib):
    rng = np.random.default_rng(4)
    M, H, I = 1, 32, 16
    t = _zeros(M, H, I, 1, 1)
    t["x"] = _rand_bf16(rng, (M, H))
    _set_code(t["w13"], t["s13"], 0, 3, 7, 0x7, 0x03)       # 6 * 3/8 * 2^-6
    _set_code(t["w13"], t["s13"], 0, I + 3, 7, 0x1, 0x05)   # 0.5 * 5/8 * 2^-6
    _set_code(t["w2"], t["s2"], 0, 11, 3, 0x9, 0x01)        # -0.5 * 2^-9
    t["gs13"][0] = 1024.0
    t["gs2"][0] = 4096.0
    out = _run(lib, t)
    xv = bits_to_f(int(t["x"][0, 7]))
    up = 1024.0 * 6 * (3 / 8) * 2.0 ** -6 * xv
    gate = 1024.0 * 0.5 * (5 / 8) * 2.0 ** -6 * xv
    h = bits_to_f(brute_bf16(silu(gate) * up))
    want = brute_bf16(4096.0 * -0.5 * 2.0 ** -9 * h)
    assert int(out[0, 11]) == want


# ---------------------------------------------------------------------------
# the layer: invariants on random NVFP4 inputs
# ---------------------------------------------------------------------------

def _random_layer(seed, M=6, H=64, I=32, E=4, top_k=3):
    from qmoe_inputs import LayerConfig, make_inputs
    cfg = LayerConfig("pin", M, H, I, E, top_k, seed)
    li = make_inputs(cfg, "cpu", weight_std=0.3)
    return dict(x=li.x.view(torch.int16).numpy().astype(np.uint16),
                w13=li.w13.numpy(), s13=li.s13.numpy(), gs13=li.gs13.numpy(),
                w2=li.w2.numpy(), s2=li.s2.numpy(), gs2=li.gs2.numpy(),
                topk_ids=li.topk_ids.numpy().copy(), topk_weights=li.topk_weights.numpy().copy())


def pin_token_permutation(lib):
    t = _random_layer(7)
    out = _run(lib, t)
    perm = np.random.default_rng(8).permutation(t["x"].shape[0])
    t2 = dict(t)
    for k in ("x", "topk_ids", "topk_weights"):
        t2[k] = np.ascontiguousarray(t[k][perm])
    out2 = _run(lib, t2)
    assert (out2 == out[perm]).all()


def pin_duplicate_expert(lib):
    """Two slots naming one expert with weights 1/2 + 1/2 equal one slot with weight 1,
    and a slot with expert -1 adds nothing."""
    t = _random_layer(9, top_k=1)
    t["topk_weights"][:] = 1.0
    _, one = _run(lib, t, return_f64=True)
    t2 = dict(t)
    t2["topk_ids"] = np.ascontiguousarray(np.repeat(t["topk_ids"], 2, axis=1))
    t2["topk_weights"] = np.full(t2["topk_ids"].shape, 0.5, np.float32)
    _, two = _run(lib, t2, return_f64=True)
    assert np.array_equal(one, two)
    t3 = dict(t)
    t3["topk_ids"] = np.ascontiguousarray(np.concatenate([np.full_like(t["topk_ids"], -1),
                                                          t["topk_ids"]], axis=1))
    t3["topk_weights"] = np.full(t3["topk_ids"].shape, 1.0, np.float32)
    _, three = _run(lib, t3, return_f64=True)
    assert np.array_equal(one, three)


def pin_weight_linearity(lib):
    t = _random_layer(10)
    _, a = _run(lib, t, return_f64=True)
    t2 = dict(t)
    t2["topk_weights"] = t["topk_weights"] * np.float32(2.0)
    _, b = _run(lib, t2, return_f64=True)
    assert np.array_equal(2.0 * a, b)
    # each slot's contribution adds: out(all slots) = sum over k of out(slot k alone)
    parts = []
    for k in range(t["topk_ids"].shape[1]):
        tk = dict(t)
        w = np.zeros_like(t["topk_weights"])
        w[:, k] = t["topk_weights"][:, k]
        tk["topk_weights"] = w
        parts.append(_run(lib, tk, return_f64=True)[1])
    assert np.allclose(sum(parts), a, rtol=1e-12, atol=1e-15)


def pin_numpy_twin(lib):
    from oracle import ref_numpy
    for seed in (12, 13):
        t = _random_layer(seed, M=5, H=64, I=48, E=3, top_k=2)
        t["topk_ids"][1, 0] = -1
        out, f64 = _run(lib, t, return_f64=True)
        twin_bf, twin64 = ref_numpy.forward(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"],
                                            t["s2"], t["gs2"], t["topk_ids"], t["topk_weights"])
        assert np.allclose(f64, twin64, rtol=1e-11, atol=1e-14)
        got = oracle.bf16_bits_to_float(out)
        assert np.array_equal(got, twin_bf)


def pin_tiny_config(lib):
    """The 4-token layer config against the NumPy statement, all tokens."""
    from oracle import ref_numpy
    from qmoe_inputs import CONFIGS, make_inputs
    li = make_inputs(CONFIGS[0], "cpu")
    t = dict(x=li.x.view(torch.int16).numpy().astype(np.uint16), w13=li.w13.numpy(),
             s13=li.s13.numpy(), gs13=li.gs13.numpy(), w2=li.w2.numpy(), s2=li.s2.numpy(),
             gs2=li.gs2.numpy(), topk_ids=li.topk_ids.numpy(), topk_weights=li.topk_weights.numpy())
    out, f64 = _run(lib, t, return_f64=True)
    twin_bf, twin64 = ref_numpy.forward(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"], t["s2"],
                                        t["gs2"], t["topk_ids"], t["topk_weights"])
    assert np.allclose(f64, twin64, rtol=1e-11, atol=1e-15)
    assert np.array_equal(oracle.bf16_bits_to_float(out), twin_bf)


def _permutation_layer(seed):
    """up[i] = x[sig(i)], gate[i] = 2 x[tau(i)] exactly, out[j] = h[pi(j)]."""
    rng = np.random.default_rng(seed)
    M, H, I, E = 3, 48, 32, 2
    t = _zeros(M, H, I, E, 2)
    t["x"] = _rand_bf16(rng, (M, H))
    sig = rng.permutation(H)[:I]
    tau = rng.permutation(H)[:I]
    pi = rng.integers(0, I, size=H)
    e = 1
    for i in range(I):
        _set_code(t["w13"], t["s13"], e, i, int(sig[i]), 0x2, 0x40)       # 1.0 * 2.0
        _set_code(t["w13"], t["s13"], e, I + i, int(tau[i]), 0x4, 0x40)   # 2.0 * 2.0
    for j in range(H):
        _set_code(t["w2"], t["s2"], e, j, int(pi[j]), 0xA, 0x30)           # -1.0 * 0.5
    t["gs13"][e] = 0.5
    t["gs2"][e] = -2.0
    t["topk_ids"][:] = [[e, -1], [-1, e], [e, 0]]
    t["topk_weights"][:] = [[1.0, 9.0], [3.0, 1.0], [1.0, 0.0]]
    return t, sig, tau, pi


def pin_swiglu_limit(lib):
    """GLM SwiGLU clamp on permutation-matrix weights: with gate = 2 x[tau(i)] and
    up = x[sig(i)] exact, h = bf16(silu(min(gate, L)) * min(max(up, -L), L)) in closed
    form, for limits that clamp many gates and ups from either side."""
    n_gate = n_up_hi = n_up_lo = 0
    for seed, L in ((31, 0.75), (32, 0.3), (33, 2.5)):
        t, sig, tau, pi = _permutation_layer(seed)
        out = _run(lib, t, swiglu_limit=L)
        for m in range(t["x"].shape[0]):
            xm = [bits_to_f(int(b)) for b in t["x"][m]]
            h = []
            for i in range(len(sig)):
                g, u = 2.0 * xm[tau[i]], xm[sig[i]]
                n_gate += g > L
                n_up_hi += u > L
                n_up_lo += u < -L
                h.append(bits_to_f(brute_bf16(silu(min(g, L)) * min(max(u, -L), L))))
            for j in range(t["x"].shape[1]):
                assert int(out[m, j]) == brute_bf16(h[pi[j]]), (seed, m, j)
    assert n_gate and n_up_hi and n_up_lo  # each clamp was exercised


def pin_swiglu_limit_infinite(lib):
    """A limit above every |gate| and |up| (or +infinity) changes nothing; a limit of 0
    or below is rejected."""
    t = _random_layer(34)
    ref, ref64 = _run(lib, t, return_f64=True)
    for L in (float("inf"), 1e30):
        out, f64 = _run(lib, t, return_f64=True, swiglu_limit=L)
        assert np.array_equal(out, ref) and np.array_equal(f64, ref64)
    for L in (0.0, -1.0, float("nan")):
        try:
            _run(lib, t, swiglu_limit=L)
        except ValueError:
            continue
        raise AssertionError(f"limit {L} accepted")


def pin_swiglu_limit_numpy_twin(lib):
    from oracle import ref_numpy
    t = _random_layer(35, M=5, H=64, I=48, E=3, top_k=2)
    for L in (0.5, 1.5):
        out, f64 = _run(lib, t, return_f64=True, swiglu_limit=L)
        twin_bf, twin64 = ref_numpy.forward(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"],
                                            t["s2"], t["gs2"], t["topk_ids"], t["topk_weights"],
                                            swiglu_limit=L)
        assert np.allclose(f64, twin64, rtol=1e-11, atol=1e-14)
        assert np.array_equal(oracle.bf16_bits_to_float(out), twin_bf)


# ---------------------------------------------------------------------------
# W4A4 variant: the activation quantizer and the layer
# ---------------------------------------------------------------------------

def _e2m1_brute(r: float) -> int:
    """Nearest E2M1 code by enumeration; ties to the even code (even mantissa)."""
    best = min(range(8), key=lambda c: (abs(abs(r) - E2M1_TABLE[c]), c & 1))
    return best | 8 if (r < 0 and best) else best


def pin_e4m3_rne(lib):
    """E4M3 rounding (round to nearest, ties to even, saturating at 448) against torch's
    float8_e4m3fn conversion of fp32-exact values, every E4M3 value onto itself, and
    the midpoints between neighbours onto the even one."""
    g = torch.Generator().manual_seed(41)
    v = torch.exp2(torch.empty(3000).uniform_(-12, 8.8, generator=g)).clamp(max=448.0)
    want = v.to(torch.float8_e4m3fn).view(torch.uint8).int().tolist()
    for a, w in zip(v.double().tolist(), want):
        assert oracle.e4m3_rne(a, lib) == w, (a, oracle.e4m3_rne(a, lib), w)
    vals = [oracle.dec_e4m3(b, lib) for b in range(0x7F)]
    for b in range(0x7F):
        assert oracle.e4m3_rne(vals[b], lib) == b
    for b in range(0x7E):
        mid = 0.5 * (vals[b] + vals[b + 1])
        assert oracle.e4m3_rne(mid, lib) == (b if b % 2 == 0 else b + 1), b
    assert oracle.e4m3_rne(1e9, lib) == 0x7E and oracle.e4m3_rne(0.0, lib) == 0


def pin_e2m1_nearest(lib):
    vals = [k / 16.0 for k in range(-128, 129)] + [7.0, -9.5, 1e-3, 5.999, 2.4999]
    for r in vals:
        assert oracle.e2m1_nearest(r, lib) == _e2m1_brute(r), r


def _nvfp4_row_brute(v):
    """Row quantizer from its definition, with torch's float8 conversion for the E4M3
    scale and enumeration for the codes."""
    v = np.asarray(v, dtype=np.float64)
    amax = float(np.abs(v).max())
    g = amax / (6.0 * 448.0) if amax > 0 else 1.0
    out = np.zeros_like(v)
    for b in range(0, v.size, 16):
        t = float(np.abs(v[b:b + 16]).max()) / 6.0 / g
        sc = float(torch.tensor([min(t, 448.0)], dtype=torch.float64).float()
                   .to(torch.float8_e4m3fn).float())
        for i in range(b, b + 16):
            if sc > 0:
                c = _e2m1_brute(v[i] / (sc * g))
                out[i] = (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7] * sc * g
    return out


def pin_nvfp4_row(lib):
    """The W4A4 activation quantizer: against the brute-force statement on random rows
    (with an all-zero block and an outlier), a fixed point on rows already in NVFP4,
    and equivariance under scaling by powers of two."""
    rng = np.random.default_rng(43)
    for n, scale in ((64, 1.0), (128, 3e-3), (256, 40.0)):
        v = rng.standard_normal(n) * scale
        v[16:32] = 0.0
        v[5] *= 30.0
        v = v.astype(np.float32).astype(np.float64)
        got = oracle.nvfp4_row(v, lib)
        assert np.array_equal(got, _nvfp4_row_brute(v)), n
        # exactly representable: codes times an E4M3 scale times g, each block holding a
        # code of magnitude 6 (so its amax / 6 / g is its scale), amax 6 * 448 * g
        g = 0.01
        codes = rng.integers(0, 16, size=n)
        codes[::16] = 7
        scales = np.array([oracle.dec_e4m3(int(b), lib) for b in rng.integers(40, 110, size=n // 16)])
        scales[0] = 448.0
        rep = np.array([oracle.dec_e2m1(int(c), lib) for c in codes]) * np.repeat(scales, 16) * g
        rep[0] = 6.0 * 448.0 * g
        assert np.array_equal(oracle.nvfp4_row(rep, lib), rep)
        for k in (-7, 5):
            assert np.array_equal(oracle.nvfp4_row(v * 2.0 ** k, lib), got * 2.0 ** k)
    assert not oracle.nvfp4_row(np.zeros(32), lib).any()


def pin_w4a4_numpy_twin(lib):
    """The W4A4 layer against the NumPy statement (ref_numpy.forward_w4a4)."""
    from oracle import ref_numpy
    for seed in (44, 45):
        t = _random_layer(seed, M=5, H=64, I=48, E=3, top_k=2)
        t["topk_ids"][2, 1] = -1
        out, f64 = oracle.forward_w4a4(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"], t["s2"],
                                       t["gs2"], t["topk_ids"], t["topk_weights"], lib=lib,
                                       nthreads=2, return_f64=True)
        twin_bf, twin64 = ref_numpy.forward_w4a4(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"],
                                                 t["s2"], t["gs2"], t["topk_ids"],
                                                 t["topk_weights"])
        assert np.allclose(f64, twin64, rtol=1e-11, atol=1e-14)
        assert np.array_equal(oracle.bf16_bits_to_float(out), twin_bf)
        # and it is a different layer from W4A16 (the quantization is not a no-op)
        w4a16 = oracle.forward(t["x"], t["w13"], t["s13"], t["gs13"], t["w2"], t["s2"],
                               t["gs2"], t["topk_ids"], t["topk_weights"], lib=lib, nthreads=2)
        assert not np.array_equal(out, w4a16)


ALL_PINS = [pin_e2m1, pin_e4m3, pin_bf16_decode, pin_bf16_round, pin_route, pin_zero_weights,
            pin_single_nibble, pin_h_given, pin_h_bound_production, pin_permutation_blocks, pin_subnormal_scale, pin_token_permutation,
            pin_duplicate_expert, pin_weight_linearity, pin_numpy_twin, pin_tiny_config,
            pin_swiglu_limit, pin_swiglu_limit_infinite, pin_swiglu_limit_numpy_twin,
            pin_e4m3_rne, pin_e2m1_nearest, pin_nvfp4_row, pin_w4a4_numpy_twin]
