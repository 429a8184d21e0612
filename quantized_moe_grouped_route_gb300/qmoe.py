"""Thin Python binding of libqmoe (ctypes): same names as the C-ABI in include/qmoe.h.

Only argument marshalling lives here: tensors become device pointers, outputs and
workspaces are allocated with torch (device memory is PyTorch's job), and every
step of the layer runs in the library's CUDA kernels.  If the library is missing
the calls raise; there is no other code path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libqmoe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "qmoe.h")

QMOE_OK = 0
QMOE_ERR_ARG = -1
QMOE_ERR_SHAPE = -2
QMOE_ERR_CUDA = -3
QMOE_ERR_TIMEOUT = -4
QMOE_ERR_ARCH = -5
QMOE_ERR_WORKSPACE = -6
QMOE_ERR_BAD_ID = -7
QMOE_FLAG_BAD_ID = 1
QMOE_FLAG_TIMEOUT = 2
QMOE_FLAG_INTERNAL = 4
QMOE_SCHED_AUTO = 0
QMOE_SCHED_DECODE = 1
QMOE_SCHED_PREFILL = 2
QMOE_SCHED_PREFILL_PAIR = 3
QMOE_W13 = 1
QMOE_W2 = 2
QMOE_SCALES_PLAIN = 0
QMOE_SCALES_SWIZZLED_128X4 = 1
QMOE_SCALES_PACKED_U32 = 2

_ERRORS = {QMOE_ERR_ARG: "argument", QMOE_ERR_SHAPE: "shape", QMOE_ERR_CUDA: "cuda",
           QMOE_ERR_TIMEOUT: "timeout", QMOE_ERR_ARCH: "arch", QMOE_ERR_WORKSPACE: "workspace",
           QMOE_ERR_BAD_ID: "bad expert id"}


class QmoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {_ERRORS.get(code, code)} ({code})")
        self.code = code


_lib = None


def lib():
    """Load libqmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libqmoe.so is missing at {LIB_PATH}: run "
                               "`python -m quantized_moe_grouped_route_gb300.build`")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def _bind(L):
    P, i32, sz, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
    sig = {
        "qmoe_sched_tile_n": (i32, [i32, i32, i32, i32]),
        "qmoe_max_tiles": (i32, [i32, i32, i32, i32]),
        "qmoe_forward_kernel_count": (i32, [i32, i32, i32, i32]),
        "qmoe_route_workspace_size": (sz, [i32, i32, i32, i32]),
        "moe_route": (i32, [P, i32, i32, i32, i32, P, P, P, P, P, P, sz, P]),
        "qmoe_repacked_fp4_size": (sz, [i32, i32, i32]),
        "qmoe_repacked_scale_size": (sz, [i32, i32, i32]),
        "moe_nvfp4_repack": (i32, [P, P, i32, i32, i32, i32, P, P, P]),
        "moe_nvfp4_repack_layout": (i32, [P, P, i32, i32, i32, i32, i32, P, P, P]),
        "qmoe_forward_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "moe_nvfp4_forward": (i32, [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P,
                                    sz, P]),
        "moe_nvfp4_forward_limit": (i32, [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                          i32, ctypes.c_float, P, sz, P]),
        "moe_nvfp4_forward_noalloc": (i32, [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                            i32, P]),
        "moe_nvfp4_forward_events": (i32, [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                           i32, P, sz, P, P]),
        "qmoe_forward_workspace_layout": (i32, [i32, i32, i32, i32, i32, i32,
                                                ctypes.POINTER(ctypes.c_size_t)]),
        "qmoe_read_error": (i32, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
        "qmoe_noalloc_read_error": (i32, [P, ctypes.POINTER(ctypes.c_uint32)]),
        "qmoe_selftest_dequant": (i32, [P, P]),
        "qmoe_selftest_timeout": (i32, [P, i64, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def exported_symbols():
    """Names of the functions the header declares (parsed from include/qmoe.h)."""
    import re
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|size_t)\s+(\w+)\s*\(", text, flags=re.M)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, rc: int):
    if rc != QMOE_OK:
        raise QmoeError(fn, rc)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: need a contiguous CUDA tensor of {dtype}, got {t.dtype} "
                         f"on {t.device}")


# --------------------------------------------------------------------- sizes
def qmoe_sched_tile_n(sched: int, M: int, top_k: int, E: int) -> int:
    return lib().qmoe_sched_tile_n(sched, M, top_k, E)


def qmoe_forward_kernel_count(M: int, top_k: int, E: int, sched: int = QMOE_SCHED_AUTO) -> int:
    return lib().qmoe_forward_kernel_count(M, top_k, E, sched)


def qmoe_max_tiles(M: int, top_k: int, E: int, tile_n: int) -> int:
    return lib().qmoe_max_tiles(M, top_k, E, tile_n)


def qmoe_route_workspace_size(M: int, top_k: int, E: int, tile_n: int) -> int:
    return lib().qmoe_route_workspace_size(M, top_k, E, tile_n)


def qmoe_forward_workspace_size(M, H, I, E, top_k, sched=QMOE_SCHED_AUTO) -> int:
    return lib().qmoe_forward_workspace_size(M, H, I, E, top_k, sched)


def qmoe_forward_workspace_layout(M, H, I, E, top_k, sched=QMOE_SCHED_AUTO) -> dict:
    arr = (ctypes.c_size_t * 10)()
    _check("qmoe_forward_workspace_layout",
           lib().qmoe_forward_workspace_layout(M, H, I, E, top_k, sched, arr))
    keys = ["offsets", "sorted_pair", "pair_pos", "tiles", "n_tiles", "xs", "h", "ypart", "total",
            "rows"]
    return dict(zip(keys, [int(v) for v in arr]))


def workspace_views(ws: torch.Tensor, M, H, I, E, top_k, sched=QMOE_SCHED_AUTO) -> dict:
    """Typed views of what a forward call left in its workspace (inspection only)."""
    L = qmoe_forward_workspace_layout(M, H, I, E, top_k, sched)
    P = M * top_k
    rows = L["rows"]

    def view(off, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype)

    return {
        "offsets": view(L["offsets"], E + 1, torch.int32),
        "sorted_pair": view(L["sorted_pair"], P, torch.int32),
        "pair_pos": view(L["pair_pos"], P, torch.int32),
        "tiles": view(L["tiles"], 3 * qmoe_max_tiles(M, top_k, E, qmoe_sched_tile_n(sched, M, top_k, E)),
                      torch.int32).view(-1, 3),
        # [2]: all tiles and, on the split prefill schedule, its first part's count
        "n_tiles": view(L["n_tiles"], 2, torch.int32),
        # the split prefill schedule's two-part tile order: the 256-byte block after the
        # counts (csrc/api.cu, forward_layout)
        "tile_order": view(L["n_tiles"] + 256,
                           qmoe_max_tiles(M, top_k, E, qmoe_sched_tile_n(sched, M, top_k, E)),
                           torch.int32),
        "xs": view(L["xs"], rows * H, torch.bfloat16).view(rows, H),
        "h": view(L["h"], rows * I, torch.bfloat16).view(rows, I),
        "ypart": view(L["ypart"], P * H, torch.float32).view(P, H),
    }


def qmoe_repacked_fp4_size(E, N, K) -> int:
    return lib().qmoe_repacked_fp4_size(E, N, K)


def qmoe_repacked_scale_size(E, N, K) -> int:
    return lib().qmoe_repacked_scale_size(E, N, K)


# --------------------------------------------------------------------- calls
def moe_route(topk_ids: torch.Tensor, E: int, tile_n: int, stream=None):
    """Returns (offsets [E+1], sorted_pair [P], pair_pos [P], tiles [max_tiles][3], n_tiles [1])."""
    _need(topk_ids, torch.int32, "topk_ids")
    M, top_k = topk_ids.shape
    dev = topk_ids.device
    P = M * top_k
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_pair = torch.empty(max(P, 1), dtype=torch.int32, device=dev)
    pair_pos = torch.empty(max(P, 1), dtype=torch.int32, device=dev)
    mt = qmoe_max_tiles(M, top_k, E, tile_n)
    if mt < 0:
        raise QmoeError("qmoe_max_tiles", mt)
    tiles = torch.empty(max(mt, 1), 3, dtype=torch.int32, device=dev)
    n_tiles = torch.empty(1, dtype=torch.int32, device=dev)
    wsb = qmoe_route_workspace_size(M, top_k, E, tile_n)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    rc = lib().moe_route(_ptr(topk_ids), M, top_k, E, tile_n, _ptr(offsets), _ptr(sorted_pair),
                         _ptr(pair_pos), _ptr(tiles), _ptr(n_tiles), _ptr(ws), wsb, _stream(stream))
    _check("moe_route", rc)
    return offsets, sorted_pair[:P], pair_pos[:P], tiles, n_tiles, ws


def moe_nvfp4_repack(w_fp4: torch.Tensor, w_scale: torch.Tensor, which: int, stream=None,
                     scale_layout: int = QMOE_SCALES_PLAIN):
    """Plain [E][N][K/2] codes + block scales -> repacked (codes, scales).  Scales are
    [E][N][K/16] bytes (QMOE_SCALES_PLAIN), N*K/16 bytes per expert in the 128x4
    swizzle of CUTLASS / FlashInfer checkpoints (QMOE_SCALES_SWIZZLED_128X4), or
    [E][N][K/64] int32 words of four scales each (QMOE_SCALES_PACKED_U32)."""
    _need(w_fp4, torch.uint8, "w_fp4")
    E, N, K2 = w_fp4.shape
    K = 2 * K2
    if scale_layout == QMOE_SCALES_PACKED_U32:
        _need(w_scale, torch.int32, "w_scale")
        if tuple(w_scale.shape) != (E, N, K // 64):
            raise ValueError("packed w_scale must be int32 [E][N][K/64]")
    else:
        _need(w_scale, torch.uint8, "w_scale")
    nbytes = w_scale.numel() * w_scale.element_size()
    if nbytes != E * N * (K // 16) or w_scale.shape[0] != E:
        raise ValueError("w_scale shape does not match w_fp4")
    if scale_layout == QMOE_SCALES_PLAIN and tuple(w_scale.shape) != (E, N, K // 16):
        raise ValueError("plain w_scale must be [E][N][K/16]")
    codes = torch.empty(qmoe_repacked_fp4_size(E, N, K), dtype=torch.uint8, device=w_fp4.device)
    scales = torch.empty(qmoe_repacked_scale_size(E, N, K), dtype=torch.uint8, device=w_fp4.device)
    rc = lib().moe_nvfp4_repack_layout(_ptr(w_fp4), _ptr(w_scale), E, N, K, which, scale_layout,
                                       _ptr(codes), _ptr(scales), _stream(stream))
    _check("moe_nvfp4_repack_layout", rc)
    return codes, scales


def moe_nvfp4_forward(x, w13_fp4, w13_scale, w13_gscale, w2_fp4, w2_scale, w2_gscale, topk_ids,
                      topk_weights, out=None, *, H: int, I: int, E: int,
                      sched: int = QMOE_SCHED_AUTO, workspace: Optional[torch.Tensor] = None,
                      stream=None, swiglu_limit: Optional[float] = None) -> torch.Tensor:
    """The layer.  w13_* / w2_* are the repacked weights from moe_nvfp4_repack.
    swiglu_limit (> 0): the GLM SwiGLU clamp (moe_nvfp4_forward_limit); None: none."""
    _need(x, torch.bfloat16, "x")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    for t, n in ((w13_fp4, "w13_fp4"), (w13_scale, "w13_scale"), (w2_fp4, "w2_fp4"),
                 (w2_scale, "w2_scale")):
        _need(t, torch.uint8, n)
    _need(w13_gscale, torch.float32, "w13_gscale")
    _need(w2_gscale, torch.float32, "w2_gscale")
    M = x.shape[0]
    top_k = topk_ids.shape[1]
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    wsb = qmoe_forward_workspace_size(M, H, I, E, top_k, sched)
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=x.device)
    if swiglu_limit is None:
        rc = lib().moe_nvfp4_forward(_ptr(x), _ptr(w13_fp4), _ptr(w13_scale), _ptr(w13_gscale),
                                     _ptr(w2_fp4), _ptr(w2_scale), _ptr(w2_gscale),
                                     _ptr(topk_ids), _ptr(topk_weights), _ptr(out), M, H, I, E,
                                     top_k, sched, _ptr(workspace), workspace.numel(),
                                     _stream(stream))
        _check("moe_nvfp4_forward", rc)
    else:
        rc = lib().moe_nvfp4_forward_limit(_ptr(x), _ptr(w13_fp4), _ptr(w13_scale),
                                           _ptr(w13_gscale), _ptr(w2_fp4), _ptr(w2_scale),
                                           _ptr(w2_gscale), _ptr(topk_ids), _ptr(topk_weights),
                                           _ptr(out), M, H, I, E, top_k, sched,
                                           float(swiglu_limit), _ptr(workspace),
                                           workspace.numel(), _stream(stream))
        _check("moe_nvfp4_forward_limit", rc)
    return out


# Size of the scratch array built into libqmoe for moe_nvfp4_forward_noalloc.
QMOE_NOALLOC_SCRATCH_BYTES = 16 << 20


def moe_nvfp4_forward_noalloc(x, w13_fp4, w13_scale, w13_gscale, w2_fp4, w2_scale, w2_gscale,
                              topk_ids, topk_weights, out, *, H: int, I: int, E: int,
                              sched: int = QMOE_SCHED_AUTO, stream=None) -> torch.Tensor:
    """The layer without a caller workspace: the library's built-in scratch array is
    used instead (for callers that cannot allocate device memory).  `out` must be
    given; nothing is allocated."""
    M = x.shape[0]
    top_k = topk_ids.shape[1]
    rc = lib().moe_nvfp4_forward_noalloc(
        _ptr(x), _ptr(w13_fp4), _ptr(w13_scale), _ptr(w13_gscale), _ptr(w2_fp4), _ptr(w2_scale),
        _ptr(w2_gscale), _ptr(topk_ids), _ptr(topk_weights), _ptr(out), M, H, I, E, top_k, sched,
        _stream(stream))
    _check("moe_nvfp4_forward_noalloc", rc)
    return out


def moe_nvfp4_forward_events(x, w13_fp4, w13_scale, w13_gscale, w2_fp4, w2_scale, w2_gscale,
                             topk_ids, topk_weights, out, events, *, H: int, I: int, E: int,
                             sched: int, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """moe_nvfp4_forward recording six torch.cuda.Event objects at the stage boundaries
    (before route, after route, gather, FC1, FC2, combine) on the launching stream."""
    M = x.shape[0]
    top_k = topk_ids.shape[1]
    arr = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    rc = lib().moe_nvfp4_forward_events(
        _ptr(x), _ptr(w13_fp4), _ptr(w13_scale), _ptr(w13_gscale), _ptr(w2_fp4), _ptr(w2_scale),
        _ptr(w2_gscale), _ptr(topk_ids), _ptr(topk_weights), _ptr(out), M, H, I, E, top_k, sched,
        _ptr(workspace), workspace.numel(), _stream(stream), arr)
    _check("moe_nvfp4_forward_events", rc)
    return out


def qmoe_read_error(workspace: torch.Tensor, stream=None):
    """(return code, flags) of the device error word at the start of a workspace."""
    flags = ctypes.c_uint32(0)
    rc = lib().qmoe_read_error(_ptr(workspace), _stream(stream), ctypes.byref(flags))
    return rc, flags.value


def qmoe_noalloc_read_error(stream=None):
    """(return code, flags) of the error word of the library's built-in scratch array
    (the last moe_nvfp4_forward_noalloc call on the current device)."""
    flags = ctypes.c_uint32(0)
    rc = lib().qmoe_noalloc_read_error(_stream(stream), ctypes.byref(flags))
    return rc, flags.value


def qmoe_selftest_dequant(device="cuda", stream=None) -> torch.Tensor:
    out = torch.empty(16 * 256 * 8, dtype=torch.int16, device=device)
    _check("qmoe_selftest_dequant", lib().qmoe_selftest_dequant(_ptr(out), _stream(stream)))
    return out


def qmoe_selftest_timeout(limit_ns: int, device="cuda", stream=None) -> int:
    ws = torch.zeros(256, dtype=torch.uint8, device=device)
    return lib().qmoe_selftest_timeout(_ptr(ws), limit_ns, _stream(stream))


class NVFP4MoE:
    """One MoE layer's repacked NVFP4 weights plus a reusable workspace."""

    def __init__(self, w13, s13, gs13, w2, s2, gs2, stream=None, scale_layout=QMOE_SCALES_PLAIN):
        E, N13, H2 = w13.shape
        self.E, self.I, self.H = E, N13 // 2, 2 * H2
        self.w13c, self.w13s = moe_nvfp4_repack(w13, s13, QMOE_W13, stream, scale_layout)
        self.w2c, self.w2s = moe_nvfp4_repack(w2, s2, QMOE_W2, stream, scale_layout)
        self.gs13 = gs13.contiguous()
        self.gs2 = gs2.contiguous()
        self._ws = None

    def workspace(self, M: int, top_k: int, sched: int = QMOE_SCHED_AUTO, device=None):
        need = qmoe_forward_workspace_size(M, self.H, self.I, self.E, top_k, sched)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8,
                                   device=device or self.w13c.device)
        return self._ws

    def __call__(self, x, topk_ids, topk_weights, out=None, sched=QMOE_SCHED_AUTO, stream=None,
                 swiglu_limit=None):
        ws = self.workspace(x.shape[0], topk_ids.shape[1], sched, x.device)
        return moe_nvfp4_forward(x, self.w13c, self.w13s, self.gs13, self.w2c, self.w2s, self.gs2,
                                 topk_ids, topk_weights, out, H=self.H, I=self.I, E=self.E,
                                 sched=sched, workspace=ws, stream=stream,
                                 swiglu_limit=swiglu_limit)
