"""The no-allocation forward entry point (moe_nvfp4_forward_noalloc).

Callers that cannot allocate device memory (a plugin inside another runtime's
enqueue step, a C host program without the process's allocator, a serving loop that
must not allocate) get the layer with the library's built-in scratch array in
place of a workspace.  Both entry points run the same kernels in the same order, so
the output must equal the regular entry point's bit for bit, on two calls in a row
(the array keeps the previous call's contents, so the second call checks that
nothing stale leaks through), including a batch just above the size where the route
keeps per-warp count tables in the scratch.  Its error word is read with
qmoe_noalloc_read_error.  This file is named to be collected last.
"""

import ctypes

import pytest
import torch

from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import CONFIGS, LayerConfig, make_inputs
from tests.helpers import check_close, oracle_forward, to_np_bf16_bits

pytestmark = pytest.mark.gpu

CASES = [
    CONFIGS[0],
    CONFIGS[1],
    # 8800 pairs: the three-kernel route, whose count tables live in the scratch
    LayerConfig("route_multi_block_m1100_h128_i128_e16_k8", 1100, 128, 128, 16, 8, seed=43),
]


def _noalloc(li, layer, cfg, out):
    return qmoe.moe_nvfp4_forward_noalloc(li.x, layer.w13c, layer.w13s, layer.gs13, layer.w2c,
                                          layer.w2s, layer.gs2, li.topk_ids, li.topk_weights, out,
                                          H=cfg.H, I=cfg.I, E=cfg.E)


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    assert qmoe.qmoe_forward_workspace_size(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k) <= \
        qmoe.QMOE_NOALLOC_SCRATCH_BYTES
    li = make_inputs(cfg, "cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    ref = layer(li.x, li.topk_ids, li.topk_weights)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        _noalloc(li, layer, cfg, out)
        rc, flags = qmoe.qmoe_noalloc_read_error()
        assert rc == qmoe.QMOE_OK and flags == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"{cfg.name}: no-alloc call {call} differs from the workspace entry point"
    if cfg.M <= 16:
        # and against the oracle directly (the workspace path's own parity tests read
        # its h back; here the outputs alone)
        check_close(to_np_bf16_bits(out), oracle_forward(li), f"{cfg.name} no-alloc vs oracle")


def test_noalloc_reports_bad_ids():
    cfg = CONFIGS[0]
    li = make_inputs(cfg, "cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    out = torch.empty(cfg.M, cfg.H, dtype=torch.bfloat16, device="cuda")
    good_ids = li.topk_ids
    li.topk_ids = good_ids.clone()
    li.topk_ids[1, 0] = cfg.E + 3      # >= E: skipped and flagged
    _noalloc(li, layer, cfg, out)
    rc, flags = qmoe.qmoe_noalloc_read_error()
    assert rc == qmoe.QMOE_ERR_BAD_ID and flags & qmoe.QMOE_FLAG_BAD_ID
    # the next call starts from a cleared error word
    li.topk_ids = good_ids
    _noalloc(li, layer, cfg, out)
    rc, flags = qmoe.qmoe_noalloc_read_error()
    assert rc == qmoe.QMOE_OK and flags == 0


def test_noalloc_rejects_batches_beyond_its_scratch():
    cfg = CONFIGS[4]  # 8192 tokens: needs gigabytes of scratch
    need = qmoe.qmoe_forward_workspace_size(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k)
    assert need > qmoe.QMOE_NOALLOC_SCRATCH_BYTES
    null = ctypes.c_void_p(0)
    rc = qmoe.lib().moe_nvfp4_forward_noalloc(null, null, null, null, null, null, null, null, null,
                                              null, cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, 0, null)
    assert rc == qmoe.QMOE_ERR_WORKSPACE
