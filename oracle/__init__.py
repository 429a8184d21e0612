"""CPU oracle for the NVFP4 W4A16 MoE layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm may import this package.  It shares no code with the CUDA path.

``qmoe_oracle.c`` is the fp64 statement of the layer (see its header for the
readings of the pages); ``ref_numpy.py`` is a second, independently structured
statement (dequantize every expert to a dense matrix, then per-expert matmuls and
a weighted sum) used to cross-check the first on small cases.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libqmoe_oracle.so")

QO_OK = 0
QO_ERR_ARG = -1
QO_ERR_NAN_SCALE = -2
QO_WARN_BAD_ID = 1


def build(force: bool = False, extra_flags=(), out_path: str | None = None) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, OpenMP)."""
    out = out_path or _LIB
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and out_path is None and os.path.exists(out) and \
            os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           *extra_flags, _SRC, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


_lib = None


def _load(path: str | None = None):
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.qo_dec_e2m1.restype = ctypes.c_double
    lib.qo_dec_e2m1.argtypes = [i32]
    lib.qo_dec_e4m3.restype = ctypes.c_double
    lib.qo_dec_e4m3.argtypes = [i32]
    lib.qo_bf16_rne.restype = ctypes.c_uint16
    lib.qo_bf16_rne.argtypes = [ctypes.c_double]
    lib.qo_bf16_to_double.restype = ctypes.c_double
    lib.qo_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.qo_route.restype = i32
    lib.qo_route.argtypes = [P, i64, i32, i32, P, P, P, P, P]
    lib.qo_forward.restype = i32
    lib.qo_forward.argtypes = [P, P, P, P, P, P, P, P, P, i64, i64, i64, i32, i32, P, i64, P, P,
                               i32]
    lib.qo_forward_hl.restype = i32
    lib.qo_forward_hl.argtypes = [P, P, P, P, P, P, P, P, P, i64, i64, i64, i32, i32, P, i64, P, P,
                                  i32, P, P, P, ctypes.c_double]
    lib.qo_forward_h.restype = i32
    lib.qo_forward_h.argtypes = [P, P, P, P, P, P, P, P, P, i64, i64, i64, i32, i32, P, i64, P, P,
                                 i32, P, P, P]
    lib.qo_e4m3_rne.restype = ctypes.c_uint8
    lib.qo_e4m3_rne.argtypes = [ctypes.c_double]
    lib.qo_e2m1_nearest.restype = i32
    lib.qo_e2m1_nearest.argtypes = [ctypes.c_double]
    lib.qo_nvfp4_row.restype = None
    lib.qo_nvfp4_row.argtypes = [P, i64]
    lib.qo_forward_w4a4.restype = i32
    lib.qo_forward_w4a4.argtypes = [P, P, P, P, P, P, P, P, P, i64, i64, i64, i32, i32, P, i64, P,
                                    P, i32]
    lib.qo_max_threads.restype = i32
    lib.qo_max_threads.argtypes = []
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(t, dtype):
    """torch tensor or array -> contiguous numpy array of `dtype` (bit view for bf16)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return np.ascontiguousarray(a)


def dec_e2m1(code: int, lib=None) -> float:
    return (lib or _load()).qo_dec_e2m1(code)


def dec_e4m3(b: int, lib=None) -> float:
    return (lib or _load()).qo_dec_e4m3(b)


def bf16_rne(v: float, lib=None) -> int:
    return (lib or _load()).qo_bf16_rne(v)


def bf16_to_double(b: int, lib=None) -> float:
    return (lib or _load()).qo_bf16_to_double(b)


def route(topk_ids, E: int, tile_n: int, lib=None):
    """Expert grouping tables; returns (offsets, sorted_pair, pair_pos, tiles[n_tiles][3], rc)."""
    ids = _np(topk_ids, np.int32).reshape(-1)
    P = ids.size
    offsets = np.zeros(E + 1, np.int32)
    sorted_pair = np.zeros(P, np.int32)
    pair_pos = np.zeros(P, np.int32)
    max_tiles = -(-P // tile_n) + E
    tiles = np.zeros((max_tiles, 3), np.int32)
    n_tiles = np.zeros(1, np.int32)
    rc = (lib or _load()).qo_route(_ptr(ids), P, E, tile_n, _ptr(offsets), _ptr(sorted_pair),
                                   _ptr(pair_pos), _ptr(tiles), _ptr(n_tiles))
    if rc < 0:
        raise ValueError(f"qo_route failed: {rc}")
    return offsets, sorted_pair, pair_pos, tiles[: int(n_tiles[0])].copy(), rc


def forward(x, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights, tokens=None,
            nthreads: int | None = None, lib=None, return_f64: bool = False, check: bool = True,
            h_given=None, return_h: bool = False, swiglu_limit: float | None = None):
    """The layer on the CPU in fp64 for `tokens` (default: all).  Returns bf16 bits as
    uint16 [n_tokens][H], plus (in this order, when asked) the fp64 values before the
    final rounding, and a dict with the h actually used ([n_tokens*top_k][I] bf16 bits)
    and the h-decision statistics.

    h_given ([n_tokens*top_k][I] bf16 bits, row t*top_k + k for the t-th listed token):
    bf16 roundings of h taken elsewhere (by the GPU); each is checked to be one of the
    two bf16 values bracketing the exact SiLU(gate)*up and then used for FC2.
    swiglu_limit (> 0, None: no clamp): gate clamped to at most the limit and up to
    [-limit, limit] before SiLU(gate)*up (the GLM form of the fc1 epilogue)."""
    lib = lib or _load()
    xb = _np(x, np.uint16)
    M, H = xb.shape
    E = int(np.asarray(w13.shape)[0])
    I = int(w13.shape[1]) // 2
    top_k = int(topk_ids.shape[1])
    a13, b13, c13 = _np(w13, np.uint8), _np(s13, np.uint8), _np(gs13, np.float32)
    a2, b2, c2 = _np(w2, np.uint8), _np(s2, np.uint8), _np(gs2, np.float32)
    ids, wts = _np(topk_ids, np.int32), _np(topk_weights, np.float32)
    if tokens is None:
        tok = None
        n = M
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        n = tok.size
    out = np.zeros((n, H), np.uint16)
    out64 = np.zeros((n, H), np.float64) if return_f64 else None
    hg = None
    if h_given is not None:
        hg = _np(h_given, np.uint16).reshape(n * top_k, I)
    stats = np.zeros(3, np.int64)
    hout = np.zeros((n * top_k, I), np.uint16) if return_h else None
    if nthreads is None:
        nthreads = lib.qo_max_threads()
    limit = float("inf") if swiglu_limit is None else float(swiglu_limit)
    rc = lib.qo_forward_hl(_ptr(xb), _ptr(a13), _ptr(b13), _ptr(c13), _ptr(a2), _ptr(b2), _ptr(c2),
                           _ptr(ids), _ptr(wts), M, H, I, E, top_k,
                           _ptr(tok) if tok is not None else None, n, _ptr(out),
                           _ptr(out64) if out64 is not None else None, nthreads,
                           _ptr(hg) if hg is not None else None, _ptr(stats),
                           _ptr(hout) if hout is not None else None, limit)
    if check and rc < 0:
        raise ValueError(f"qo_forward failed: {rc}")
    res = [out]
    if return_f64:
        res.append(out64)
    if return_h or h_given is not None:
        res.append({"h": hout, "compared": int(stats[0]), "flipped": int(stats[1]),
                    "outside": int(stats[2])})
    return tuple(res) if len(res) > 1 else out


def e4m3_rne(v: float, lib=None) -> int:
    """E4M3 byte nearest to v >= 0, ties to even, saturating at 448."""
    return (lib or _load()).qo_e4m3_rne(v)


def e2m1_nearest(r: float, lib=None) -> int:
    """E2M1 code nearest to r, ties to the even mantissa, saturating at 6."""
    return (lib or _load()).qo_e2m1_nearest(r)


def nvfp4_row(v, lib=None) -> np.ndarray:
    """NVFP4 encode-decode of activation rows (last axis, a multiple of 16), as the W4A4
    variant quantizes x and h (see qo_forward_w4a4)."""
    a = np.array(v, dtype=np.float64, copy=True)
    rows = a.reshape(-1, a.shape[-1])
    for r in rows:
        (lib or _load()).qo_nvfp4_row(_ptr(r), r.size)
    return rows.reshape(a.shape)


def forward_w4a4(x, w13, s13, gs13, w2, s2, gs2, topk_ids, topk_weights, tokens=None,
                 nthreads: int | None = None, lib=None, return_f64: bool = False):
    """The W4A4 variant of the layer (x and h quantized to NVFP4 per row, see
    qo_forward_w4a4) on the CPU in fp64; bf16 bits [n_tokens][H] (and the fp64 values)."""
    lib = lib or _load()
    xb = _np(x, np.uint16)
    M, H = xb.shape
    E = int(np.asarray(w13.shape)[0])
    I = int(w13.shape[1]) // 2
    top_k = int(topk_ids.shape[1])
    a13, b13, c13 = _np(w13, np.uint8), _np(s13, np.uint8), _np(gs13, np.float32)
    a2, b2, c2 = _np(w2, np.uint8), _np(s2, np.uint8), _np(gs2, np.float32)
    ids, wts = _np(topk_ids, np.int32), _np(topk_weights, np.float32)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = M if tok is None else tok.size
    out = np.zeros((n, H), np.uint16)
    out64 = np.zeros((n, H), np.float64) if return_f64 else None
    rc = lib.qo_forward_w4a4(_ptr(xb), _ptr(a13), _ptr(b13), _ptr(c13), _ptr(a2), _ptr(b2),
                             _ptr(c2), _ptr(ids), _ptr(wts), M, H, I, E, top_k,
                             _ptr(tok) if tok is not None else None, n, _ptr(out),
                             _ptr(out64) if out64 is not None else None,
                             nthreads or lib.qo_max_threads())
    if rc < 0:
        raise ValueError(f"qo_forward_w4a4 failed: {rc}")
    return (out, out64) if return_f64 else out


def max_threads(lib=None) -> int:
    return (lib or _load()).qo_max_threads()


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    u = (bits.astype(np.uint32) << 16).view(np.float32)
    return u.astype(np.float64)
