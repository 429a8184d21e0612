"""GB300-native NVFP4 W4A16 mixture-of-experts layer.

The layer runs in hand-written sm_103a CUDA kernels behind a C-ABI shared library
(``include/qmoe.h``, ``_lib/libqmoe.so``); ``qmoe`` is its thin ctypes binding.
"""

from .qmoe import (  # noqa: F401
    NVFP4MoE, QmoeError, moe_nvfp4_forward, moe_nvfp4_repack, moe_route, qmoe_forward_workspace_size,
    qmoe_max_tiles, qmoe_read_error, qmoe_repacked_fp4_size, qmoe_repacked_scale_size,
    qmoe_route_workspace_size, qmoe_sched_tile_n, qmoe_selftest_dequant, qmoe_selftest_timeout,
    QMOE_SCHED_AUTO, QMOE_SCHED_DECODE, QMOE_SCHED_PREFILL, QMOE_SCHED_PREFILL_PAIR, QMOE_W13,
    QMOE_W2, QMOE_SCALES_PLAIN, QMOE_SCALES_SWIZZLED_128X4)
