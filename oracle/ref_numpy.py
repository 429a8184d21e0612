"""Second CPU statement of the NVFP4 W4A16 MoE layer, in NumPy float64.

Test infrastructure only (see the package docstring).  Structured like the
dequantize-then-linear statement on the tilelang_kernels.py page (grouped_gemm_fp4):
every expert matrix is first expanded to a dense float64 matrix, then each expert's
tokens go through FC1, SwiGLU, FC2 as matrix products, and the routing-weighted
outputs are summed over the top-k slots.  The format decoders here are written
from the bit-field definitions (no lookup table), independently of the C oracle,
so that the two statements cross-check each other.  Meant for small shapes.
"""

from __future__ import annotations

import numpy as np


def e2m1_values(codes: np.ndarray) -> np.ndarray:
    """E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit) -> float64."""
    c = codes.astype(np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m * 0.5, e - 1))
    return np.where(s == 1, -mag, mag)


def e4m3_values(b: np.ndarray) -> np.ndarray:
    """E4M3 (fn variant) bit patterns -> float64; 0x7F / 0xFF give NaN."""
    b = b.astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), as float64."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    mant, ex = np.frexp(a)                      # a = mant * 2^ex, mant in [0.5, 1)
    e = np.maximum(ex - 1, -126)                # normal exponent, clamped to the subnormal one
    q = np.ldexp(np.ones_like(a), e - 7)        # spacing of bf16 values near a
    r = np.rint(a / q) * q                      # numpy rint: ties to even
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    r = np.where(a == 0, 0.0, r)
    return np.copysign(r, v)


def dequant(w: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Plain [..., N, K/2] codes + [..., N, K/16] scales -> dense float64 [..., N, K]."""
    lo = w & 0xF
    hi = w >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*w.shape[:-1], w.shape[-1] * 2)
    vals = e2m1_values(codes)
    sc = np.repeat(e4m3_values(s), 16, axis=-1)
    return vals * sc


def forward(x_bf16_bits, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights, swiglu_limit=None):
    """Returns the layer output [M][H] as float64 values of bf16 numbers, plus the
    float64 sum before the final rounding.  swiglu_limit (None: none) clamps gate from
    above and up to [-limit, limit] before SiLU(gate) * up."""
    x = (np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    x = x.astype(np.float64)
    M, H = x.shape
    E = w13.shape[0]
    I = w13.shape[1] // 2
    top_k = topk_ids.shape[1]
    acc = np.zeros((M, H), np.float64)
    for e in range(E):
        toks, slots = np.nonzero(topk_ids == e)
        if toks.size == 0:
            continue
        W13 = dequant(w13[e], s13[e]) * np.float64(gs13[e])   # [2I][H]
        W2 = dequant(w2[e], s2[e]) * np.float64(gs2[e])       # [H][I]
        g = x[toks] @ W13.T                                   # [n][2I]
        up, gate = g[:, :I], g[:, I:]
        if swiglu_limit is not None:
            gate = np.minimum(gate, swiglu_limit)
            up = np.clip(up, -swiglu_limit, swiglu_limit)
        h = round_bf16(gate / (1.0 + np.exp(-gate)) * up)
        y = h @ W2.T                                          # [n][H]
        contrib = y * topk_weights[toks, slots].astype(np.float64)[:, None]
        # add slot by slot in ascending k so each token's sum runs in k order
        for k in range(top_k):
            sel = slots == k
            np.add.at(acc, toks[sel], contrib[sel])
    return round_bf16(acc), acc


def nvfp4_rows(v: np.ndarray) -> np.ndarray:
    """NVFP4 encode-decode of activation rows (last axis, a multiple of 16) as the W4A4
    variant defines it: per row g = amax / (6 * 448) (1 for an all-zero row); per
    16-block the E4M3 scale nearest (ties to even) to blockamax / 6 / g; each value the
    E2M1 value nearest (ties to the even mantissa, at most 6) to v / (scale * g), times
    scale * g.  Written with NumPy array operations."""
    v = np.asarray(v, dtype=np.float64)
    shp = v.shape
    rows = v.reshape(-1, shp[-1])
    amax = np.abs(rows).max(axis=1, keepdims=True)
    g = np.where(amax > 0, amax / (6.0 * 448.0), 1.0)
    blk = rows.reshape(rows.shape[0], -1, 16)
    bmax = np.abs(blk).max(axis=2, keepdims=True)
    t = bmax / 6.0 / g[:, :, None]
    # E4M3: 3 mantissa bits, exponents down to -6 (subnormal spacing 2^-9), max 448
    e = np.floor(np.log2(np.where(t > 0, t, 1.0)))
    q = np.exp2(np.maximum(e, -6.0) - 3.0)
    sc = np.minimum(np.rint(t / q) * q, 448.0)
    sc = np.where(t > 0, sc, 0.0)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    r = np.abs(blk) / np.where(sc > 0, sc * g[:, :, None], 1.0)
    d = np.abs(r[..., None] - mags)                      # distance to each magnitude
    # nearest; on a tie the even code index (even mantissa) wins: add a tiny bias to odd
    best = np.argmin(d + (np.arange(8) % 2) * 1e-12 * np.maximum(r[..., None], 1.0), axis=-1)
    out = np.sign(blk) * mags[best] * sc * g[:, :, None]
    out = np.where(sc > 0, out, 0.0)
    return out.reshape(shp)


def forward_w4a4(x_bf16_bits, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights):
    """The W4A4 variant: x quantized per token and h (after its bf16 rounding) per pair
    with nvfp4_rows, otherwise as forward()."""
    x = (np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    x = nvfp4_rows(x.astype(np.float64))
    M, H = x.shape
    E = w13.shape[0]
    top_k = topk_ids.shape[1]
    I = w13.shape[1] // 2
    acc = np.zeros((M, H), np.float64)
    for e in range(E):
        toks, slots = np.nonzero(topk_ids == e)
        if toks.size == 0:
            continue
        W13 = dequant(w13[e], s13[e]) * np.float64(gs13[e])
        W2 = dequant(w2[e], s2[e]) * np.float64(gs2[e])
        g = x[toks] @ W13.T
        up, gate = g[:, :I], g[:, I:]
        h = nvfp4_rows(round_bf16(gate / (1.0 + np.exp(-gate)) * up))
        contrib = (h @ W2.T) * topk_weights[toks, slots].astype(np.float64)[:, None]
        for k in range(top_k):
            sel = slots == k
            np.add.at(acc, toks[sel], contrib[sel])
    return round_bf16(acc), acc
