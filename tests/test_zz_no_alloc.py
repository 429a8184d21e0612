"""The no-allocation forward entry point (moe_nvfp4_forward_noalloc).

Callers that cannot allocate device memory (a plugin inside another runtime's
enqueue step, a C host program without the process's allocator, a serving loop that
must not allocate) get the layer with the library's built-in scratch array in
place of a workspace.  Its output must match the regular entry point's, within the
layer tolerance, on two calls in a row (the array keeps the previous call's
contents, so the second call checks that nothing stale leaks through).  This file
is named to be collected last.
"""

import ctypes

import pytest
import torch

from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import CONFIGS, make_inputs
from tests.helpers import check_close, to_np_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [CONFIGS[0], CONFIGS[1]], ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    li = make_inputs(cfg, "cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    ref = layer(li.x, li.topk_ids, li.topk_weights)
    torch.cuda.synchronize()
    ref_bits = to_np_bf16_bits(ref)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        qmoe.moe_nvfp4_forward_noalloc(li.x, layer.w13c, layer.w13s, layer.gs13, layer.w2c,
                                       layer.w2s, layer.gs2, li.topk_ids, li.topk_weights, out,
                                       H=cfg.H, I=cfg.I, E=cfg.E)
        torch.cuda.synchronize()
        check_close(to_np_bf16_bits(out), ref_bits, f"{cfg.name} no-alloc call {call}")


def test_noalloc_rejects_batches_beyond_its_scratch():
    cfg = CONFIGS[4]  # 8192 tokens: needs gigabytes of scratch
    need = qmoe.qmoe_forward_workspace_size(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k)
    assert need > qmoe.QMOE_NOALLOC_SCRATCH_BYTES
    null = ctypes.c_void_p(0)
    rc = qmoe.lib().moe_nvfp4_forward_noalloc(null, null, null, null, null, null, null, null, null,
                                              null, cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, 0, null)
    assert rc == qmoe.QMOE_ERR_WORKSPACE
