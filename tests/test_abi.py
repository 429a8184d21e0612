"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every
symbol include/qmoe.h declares, answers the size queries, and rejects bad
arguments before touching the device."""

import ctypes

import pytest

from quantized_moe_grouped_route_gb300 import qmoe


@pytest.fixture(scope="module")
def lib():
    from quantized_moe_grouped_route_gb300 import build
    build.build()
    return qmoe.lib()


def test_exports_every_declared_symbol(lib):
    names = qmoe.exported_symbols()
    assert "moe_route" in names and "moe_nvfp4_forward" in names and "moe_nvfp4_repack" in names
    for n in names:
        assert hasattr(lib, n), n


def test_size_queries(lib):
    assert qmoe.qmoe_max_tiles(16, 8, 256, 32) == 4 + 256
    assert qmoe.qmoe_max_tiles(8192, 8, 256, 256) == 256 + 256
    assert qmoe.qmoe_sched_tile_n(qmoe.QMOE_SCHED_AUTO, 16, 8, 256) == 16
    assert qmoe.qmoe_sched_tile_n(qmoe.QMOE_SCHED_AUTO, 8192, 8, 256) == 320
    # experts averaging fewer than 192 pairs: the narrow prefill tiles
    assert qmoe.qmoe_sched_tile_n(qmoe.QMOE_SCHED_AUTO, 2048, 8, 128) == 192
    assert qmoe.qmoe_sched_tile_n(qmoe.QMOE_SCHED_PREFILL, 16, 8, 256) == 192
    assert qmoe.qmoe_sched_tile_n(qmoe.QMOE_SCHED_PREFILL_PAIR, 8192, 8, 256) == 256
    # above 8192 pairs the route keeps per-warp count tables in its workspace
    assert qmoe.qmoe_route_workspace_size(1024, 8, 256, 320) == 256
    # the multi-block route's per-warp count tables and one bad-id flag per block
    assert qmoe.qmoe_route_workspace_size(8192, 8, 256, 320) == 256 + 16 * (16 * 256 + 1) * 4
    # kernels per forward: route (one, or three above 8192 pairs), gather, FC1, FC2, combine
    assert qmoe.qmoe_forward_kernel_count(16, 8, 256, qmoe.QMOE_SCHED_AUTO) == 5
    assert qmoe.qmoe_forward_kernel_count(8192, 8, 256, qmoe.QMOE_SCHED_AUTO) == 7
    # experts averaging fewer than 192 pairs: FC1 and FC2 as two launches each (tiles of
    # more than 64 pairs, then the others)
    assert qmoe.qmoe_forward_kernel_count(2048, 8, 128, qmoe.QMOE_SCHED_AUTO) == 9
    assert qmoe.qmoe_forward_kernel_count(512, 8, 128, qmoe.QMOE_SCHED_AUTO) == 7
    assert qmoe.qmoe_forward_kernel_count(0, 8, 256, qmoe.QMOE_SCHED_AUTO) == 0
    assert qmoe.qmoe_forward_kernel_count(4, 0, 8, qmoe.QMOE_SCHED_AUTO) == qmoe.QMOE_ERR_ARG
    assert qmoe.qmoe_repacked_fp4_size(256, 4096, 7168) == 256 * 4096 * 3584
    assert qmoe.qmoe_repacked_scale_size(256, 7168, 2048) == 256 * 7168 * 128
    ws = qmoe.qmoe_forward_workspace_size(8192, 7168, 2048, 256, 8)
    P = 8192 * 8
    # gathered activations, h and fp32 partials dominate
    assert ws >= P * 7168 * 2 + P * 2048 * 2 + P * 7168 * 4
    assert qmoe.qmoe_forward_workspace_size(4, 100, 128, 8, 2) == 0  # bad shape


def test_bad_arguments_are_rejected_before_any_device_work(lib):
    null = ctypes.c_void_p(0)
    # H not a multiple of 128
    rc = lib.moe_nvfp4_forward(null, null, null, null, null, null, null, null, null, null,
                               4, 100, 128, 8, 2, 0, null, 0, null)
    assert rc == qmoe.QMOE_ERR_SHAPE
    # E out of range
    rc = lib.moe_nvfp4_forward(null, null, null, null, null, null, null, null, null, null,
                               4, 128, 128, 0, 2, 0, null, 0, null)
    assert rc == qmoe.QMOE_ERR_SHAPE
    # null pointers
    rc = lib.moe_nvfp4_forward(null, null, null, null, null, null, null, null, null, null,
                               4, 128, 128, 8, 2, 0, null, 0, null)
    assert rc == qmoe.QMOE_ERR_ARG
    # bad schedule
    rc = lib.moe_nvfp4_forward(null, null, null, null, null, null, null, null, null, null,
                               4, 128, 128, 8, 2, 7, null, 0, null)
    assert rc == qmoe.QMOE_ERR_ARG
    # zero tokens is a no-op that succeeds without touching anything
    rc = lib.moe_nvfp4_forward(null, null, null, null, null, null, null, null, null, null,
                               0, 128, 128, 8, 2, 0, null, 0, null)
    assert rc == qmoe.QMOE_OK
    # SwiGLU limit: zero, negative or NaN rejected before anything else is looked at
    # (zero tokens included); +infinity and positive limits pass to the pointer checks
    for bad in (0.0, -1.0, float("nan")):
        for M in (4, 0):
            rc = lib.moe_nvfp4_forward_limit(null, null, null, null, null, null, null, null, null,
                                             null, M, 128, 128, 8, 2, 0, bad, null, 0, null)
            assert rc == qmoe.QMOE_ERR_ARG, (bad, M)
    for good in (float("inf"), 7.0):
        rc = lib.moe_nvfp4_forward_limit(null, null, null, null, null, null, null, null, null,
                                         null, 0, 128, 128, 8, 2, 0, good, null, 0, null)
        assert rc == qmoe.QMOE_OK
    # repack with a scale layout: unknown layout, then the same checks as the plain call
    assert lib.moe_nvfp4_repack_layout(null, null, 1, 128, 128, 1, 2, null, null, null) == \
        qmoe.QMOE_ERR_ARG
    assert lib.moe_nvfp4_repack_layout(null, null, 1, 100, 128, 1, 1, null, null, null) == \
        qmoe.QMOE_ERR_SHAPE
    assert lib.moe_nvfp4_repack_layout(null, null, 1, 128, 128, 1, 1, null, null, null) == \
        qmoe.QMOE_ERR_ARG
    # repack: bad role, bad shape
    assert lib.moe_nvfp4_repack(null, null, 1, 128, 128, 3, null, null, null) == qmoe.QMOE_ERR_ARG
    assert lib.moe_nvfp4_repack(null, null, 1, 100, 128, 1, null, null, null) == qmoe.QMOE_ERR_SHAPE
    # route: bad tile height, null outputs
    assert lib.moe_route(null, 4, 2, 8, 0, null, null, null, null, null, null, 256, null) == \
        qmoe.QMOE_ERR_SHAPE
    assert lib.moe_route(null, 4, 2, 8, 16, null, null, null, null, null, null, 256, null) == \
        qmoe.QMOE_ERR_ARG
    # error-word read and diagnostics with null pointers
    flags = ctypes.c_uint32(0)
    assert lib.qmoe_read_error(null, null, ctypes.byref(flags)) == qmoe.QMOE_ERR_ARG
    assert lib.qmoe_selftest_dequant(null, null) == qmoe.QMOE_ERR_ARG
    assert lib.qmoe_selftest_timeout(null, 1000000, null) == qmoe.QMOE_ERR_ARG
