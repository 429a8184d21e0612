"""GPU parity of the GLM SwiGLU limit (moe_nvfp4_forward_limit) against the CPU
oracle: gate clamped from above and up to [-limit, limit] before SiLU(gate) * up
(megamoe_rm.cu page, fc1_rm epilogue).  Same checks as the plain layer: every GPU h
value a valid bf16 rounding of the oracle's exact clamped value, outputs within
|got - ref| <= 2e-2 |ref| + 2e-3 rms(ref) of the oracle fed those h decisions."""

import numpy as np
import pytest
import torch

from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import CONFIGS, LayerConfig, make_inputs
from tests.helpers import check_layer, forced_tokens, gpu_forward

pytestmark = pytest.mark.gpu

SCHEDS = [qmoe.QMOE_SCHED_DECODE, qmoe.QMOE_SCHED_PREFILL, qmoe.QMOE_SCHED_PREFILL_PAIR]

# name, M, H, I, E, top_k: decode-sized, narrow prefill tiles, a two-chain wide tile
SHAPES = [
    ("m37_h256_i256_e5_k3", 37, 256, 256, 5, 3),
    ("m129_h512_i256_e16_k4", 129, 512, 256, 16, 4),
    ("m580_h256_i128_e2_k1", 580, 256, 128, 2, 1),
]


def _clamped_share(li, limit):
    """Share of (pair, intermediate) gate and up values the limit changes, from the
    dense fp64 pre-activations of a few tokens (to show the test exercises the clamp)."""
    from oracle import ref_numpy
    x = li.x[:8].cpu().view(torch.int16).numpy().astype(np.uint16)
    xf = ((x.astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
    e = int(li.topk_ids[0, 0])
    w = ref_numpy.dequant(li.w13[e].cpu().numpy(), li.s13[e].cpu().numpy()) * float(li.gs13[e])
    g = xf @ w.T
    I = w.shape[0] // 2
    return float(np.mean(g[:, I:] > limit)), float(np.mean(np.abs(g[:, :I]) > limit))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s[0])
@pytest.mark.parametrize("sched", SCHEDS)
def test_small_shapes_with_limit(shape, sched):
    name, M, H, I, E, k = shape
    li = make_inputs(LayerConfig(name, M, H, I, E, k, seed=23), "cpu").to("cuda")
    limit = 0.2
    gate_share, up_share = _clamped_share(li, limit)
    assert gate_share > 0.05 and up_share > 0.1
    out, layer = gpu_forward(li, sched, swiglu_limit=limit)
    check_layer(li, out, layer._ws, sched, what=f"{name} sched={sched} limit={limit}",
                swiglu_limit=limit)


@pytest.mark.parametrize("cfg", [CONFIGS[1], CONFIGS[3], CONFIGS[4]], ids=lambda c: c.name)
def test_full_configs_with_limit_sampled_tokens(cfg):
    li = make_inputs(cfg, "cuda")
    limit = 1.0
    out, layer = gpu_forward(li, qmoe.QMOE_SCHED_AUTO, swiglu_limit=limit)
    rc, flags = qmoe.qmoe_read_error(layer._ws)
    assert rc == 0 and flags == 0
    toks = forced_tokens(li, qmoe.QMOE_SCHED_AUTO, n_random=32, seed=cfg.seed)
    check_layer(li, out, layer._ws, qmoe.QMOE_SCHED_AUTO, tokens=toks,
                what=f"{cfg.name} limit={limit}", swiglu_limit=limit)
    # deterministic
    out2, _ = gpu_forward(li, qmoe.QMOE_SCHED_AUTO, layer, swiglu_limit=limit)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("sched", SCHEDS)
def test_infinite_limit_is_the_plain_layer(sched):
    li = make_inputs(LayerConfig("m300_h384_i128_e3_k2", 300, 384, 128, 3, 2, seed=29),
                     "cpu").to("cuda")
    plain, layer = gpu_forward(li, sched)
    plain = plain.clone()
    inf, _ = gpu_forward(li, sched, layer, swiglu_limit=float("inf"))
    assert torch.equal(plain.view(torch.int16), inf.view(torch.int16))
    # a limit above every |gate| and |up| gives the plain layer's values as well
    big, _ = gpu_forward(li, sched, layer, swiglu_limit=1e30)
    assert torch.equal(plain.view(torch.int16), big.view(torch.int16))


def test_bad_limit_is_rejected():
    li = make_inputs(CONFIGS[0], "cpu").to("cuda")
    for bad in (0.0, -0.5, float("nan")):
        with pytest.raises(qmoe.QmoeError):
            gpu_forward(li, qmoe.QMOE_SCHED_AUTO, swiglu_limit=bad)
