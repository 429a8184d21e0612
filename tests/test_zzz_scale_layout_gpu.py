"""GPU: the repack reads block scales in the 128x4 swizzle of CUTLASS / FlashInfer
NVFP4 checkpoints (megamoe_rm.cu page, scale_off) and as uint32 words of four scales
(tilelang_kernels.py page, grouped_gemm_fp4_packed_sf), and writes exactly the bytes
it writes from the same scales in plain row-major order; a layer built from either
gives bit-identical outputs."""

import numpy as np
import pytest
import torch

from oracle import scale_layout
from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _swizzled(s: torch.Tensor) -> torch.Tensor:
    sw = scale_layout.swizzle_128x4(s.cpu().numpy())
    return torch.from_numpy(np.ascontiguousarray(sw)).to(s.device)


def _packed(s: torch.Tensor) -> torch.Tensor:
    pk = scale_layout.pack_u32(s.cpu().numpy()).view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(pk)).to(s.device)


@pytest.mark.parametrize("which", [qmoe.QMOE_W13, qmoe.QMOE_W2])
@pytest.mark.parametrize("E,N,K", [(3, 256, 384), (2, 128, 128), (1, 384, 1024)])
def test_swizzled_scales_repack_to_the_same_bytes(which, E, N, K):
    g = torch.Generator(device="cuda").manual_seed(E * 1000 + N + K + which)
    w = torch.randint(0, 256, (E, N, K // 2), generator=g, device="cuda", dtype=torch.int32)
    s = torch.randint(0, 256, (E, N, K // 16), generator=g, device="cuda", dtype=torch.int32)
    w, s = w.to(torch.uint8), s.to(torch.uint8)
    c0, s0 = qmoe.moe_nvfp4_repack(w, s, which)
    c1, s1 = qmoe.moe_nvfp4_repack(w, _swizzled(s), which,
                                   scale_layout=qmoe.QMOE_SCALES_SWIZZLED_128X4)
    c2, s2 = qmoe.moe_nvfp4_repack(w, _packed(s), which, scale_layout=qmoe.QMOE_SCALES_PACKED_U32)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1) and torch.equal(c0, c2)
    assert torch.equal(s0, s1) and torch.equal(s0, s2)


def test_layer_from_swizzled_or_packed_scales_is_bit_identical():
    li = make_inputs(CONFIGS[0], "cpu").to("cuda")
    plain = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    swz = qmoe.NVFP4MoE(li.w13, _swizzled(li.s13), li.gs13, li.w2, _swizzled(li.s2), li.gs2,
                        scale_layout=qmoe.QMOE_SCALES_SWIZZLED_128X4)
    pkd = qmoe.NVFP4MoE(li.w13, _packed(li.s13), li.gs13, li.w2, _packed(li.s2), li.gs2,
                        scale_layout=qmoe.QMOE_SCALES_PACKED_U32)
    a = plain(li.x, li.topk_ids, li.topk_weights)
    b = swz(li.x, li.topk_ids, li.topk_weights)
    c = pkd(li.x, li.topk_ids, li.topk_weights)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
