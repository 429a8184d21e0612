"""GPU parity of the whole layer (moe_nvfp4_forward through the C-ABI) against the
CPU oracle: small shapes element by element, the five workload configs at full
size on sampled tokens (the benchmark's launch configuration), edge cases and
determinism.  Tolerance per element: |got - ref| <= 2e-2 |ref| + 2e-3 rms(ref)."""

import pytest
import torch

from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import CONFIGS, LayerConfig, make_inputs
from tests.helpers import check_layer, forced_tokens, gpu_forward

pytestmark = pytest.mark.gpu

SCHEDS = [qmoe.QMOE_SCHED_DECODE, qmoe.QMOE_SCHED_PREFILL, qmoe.QMOE_SCHED_PREFILL_PAIR,
          qmoe.QMOE_SCHED_AUTO]


@pytest.mark.parametrize("sched", SCHEDS)
def test_tiny_config_all_tokens(sched):
    li = make_inputs(CONFIGS[0], "cpu").to("cuda")
    out, layer = gpu_forward(li, sched)
    check_layer(li, out, layer._ws, sched, what=f"tiny sched={sched}")


SMALL = [
    # name, M, H, I, E, top_k: several tiles per expert, ragged tails, one expert
    ("m37_h256_i256_e5_k3", 37, 256, 256, 5, 3),
    ("m300_h384_i128_e3_k2", 300, 384, 128, 3, 2),
    ("m70_h128_i384_e1_k1", 70, 128, 384, 1, 1),
    ("m129_h512_i256_e16_k4", 129, 512, 256, 16, 4),
    # experts of 257..320 pairs (one two-chain prefill tile) and of more (a tail tile)
    ("m580_h256_i128_e2_k1", 580, 256, 128, 2, 1),
    ("m700_h256_i256_e2_k1", 700, 256, 256, 2, 1),
    # decode schedule, stream-K: fewer K steps than CTAs (units split over up to four
    # CTAs, most CTAs idle) and a few steps per CTA (units split over many CTAs)
    ("sk_m1_h1024_i1024_e4_k1", 1, 1024, 1024, 4, 1),
    ("sk_m3_h7168_i512_e2_k2", 3, 7168, 512, 2, 2),
    # decode schedule with more than two FC1 units per CTA (about 500 units of 4 steps on
    # 152 SMs), split: most CTAs start and end inside a unit
    ("sk_m16_h1024_i2048_e16_k8", 16, 1024, 2048, 16, 8),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s[0])
@pytest.mark.parametrize("sched", SCHEDS[:3])
def test_small_shapes_all_tokens(shape, sched):
    name, M, H, I, E, k = shape
    li = make_inputs(LayerConfig(name, M, H, I, E, k, seed=17), "cpu").to("cuda")
    # some slots without an expert
    ids = li.topk_ids.clone()
    ids[::7, 0] = -1
    li.topk_ids = ids.contiguous()
    out, layer = gpu_forward(li, sched)
    check_layer(li, out, layer._ws, sched, what=f"{name} sched={sched}")


@pytest.mark.parametrize("name,sched", [("sk_m16_h1024_i2048_e16_k8", qmoe.QMOE_SCHED_DECODE),
                                        ("sk_m1_h1024_i1024_e4_k1", qmoe.QMOE_SCHED_DECODE),
                                        ("m300_h384_i128_e3_k2", qmoe.QMOE_SCHED_PREFILL)])
def test_forward_needs_no_zeroed_workspace(name, sched):
    """The forward zeroes what it needs itself (the error word and the decode schedule's
    split-unit counters, in the route): a workspace full of garbage gives the same bits
    as a zeroed one, and a clean error word."""
    _, M, H, I, E, k = next(s for s in SMALL if s[0] == name)
    li = make_inputs(LayerConfig(name, M, H, I, E, k, seed=29), "cpu").to("cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    ws = layer.workspace(M, k, sched, "cuda")
    outs = []
    for fill in (0x00, 0xA5, 0xFF):
        ws.fill_(fill)
        out = qmoe.moe_nvfp4_forward(li.x, layer.w13c, layer.w13s, layer.gs13, layer.w2c,
                                     layer.w2s, layer.gs2, li.topk_ids, li.topk_weights,
                                     H=H, I=I, E=E, sched=sched, workspace=ws)
        torch.cuda.synchronize()
        assert qmoe.qmoe_read_error(ws) == (qmoe.QMOE_OK, 0), (name, fill)
        outs.append(out)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


# Expert loads around the split prefill schedule's boundaries: tiles of up to 192 pairs,
# those of at most 64 pairs on the decode pipeline, the rest on the prefill kernel.
SPLIT_LOADS = [0, 1, 15, 16, 17, 63, 64, 65, 100, 128, 191, 192, 193, 256, 257, 300]


# Every expert between 65 and 192 pairs: the split schedule's second launch has no tiles.
SPLIT_LOADS_WIDE = [65, 66, 80, 100, 127, 150, 191, 192, 70, 91]


@pytest.mark.parametrize("H,I,loads", [(256, 128, SPLIT_LOADS), (384, 384, SPLIT_LOADS),
                                       (256, 128, SPLIT_LOADS_WIDE)],
                         ids=["h256_i128", "h384_i384", "h256_i128_all_wide"])
def test_split_prefill_tile_sizes(H, I, loads):
    """Every expert load of SPLIT_LOADS in one layer (1858 pairs over 16 experts, so the
    prefill schedule splits its tiles): both parts of the tile order are non-empty and
    every tile size at the boundaries occurs; with I = 384 FC2's last K step holds one
    of its two 128-wide blocks.  SPLIT_LOADS_WIDE leaves the second part empty."""
    E, k = len(loads), 2
    flat = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(loads)])
    g = torch.Generator().manual_seed(23)
    flat = flat[torch.randperm(flat.numel(), generator=g)]
    M = flat.numel() // k
    cfg = LayerConfig(f"split_h{H}_i{I}", M, H, I, E, k, seed=29)
    li = make_inputs(cfg, "cpu")
    li.topk_ids = flat[: M * k].view(M, k).contiguous()
    li = li.to("cuda")
    # route (one block), gather, two FC1 and two FC2 launches, combine
    assert qmoe.qmoe_forward_kernel_count(M, k, E, qmoe.QMOE_SCHED_PREFILL) == 7
    for sched in (qmoe.QMOE_SCHED_AUTO, qmoe.QMOE_SCHED_PREFILL):
        out, layer = gpu_forward(li, sched)
        check_layer(li, out, layer._ws, sched, what=f"split H={H} I={I} sched={sched}")
        again, _ = gpu_forward(li, sched, layer=layer)
        assert torch.equal(out, again), "the split schedule must be deterministic"


def _tile_order_of(li, sched):
    out, layer = gpu_forward(li, sched)
    M, k = li.topk_ids.shape
    c = li.cfg
    v = qmoe.workspace_views(layer._ws, M, c.H, c.I, c.E, k, sched)
    nt, nwide = (int(x) for x in v["n_tiles"].cpu())
    return v["tiles"][:nt].cpu().numpy(), v["tile_order"][:nt].cpu().numpy(), nwide


@pytest.mark.parametrize("case", ["mixed", "all_wide", "multi_block_route"])
def test_split_tile_order(case):
    """The route's two-part tile order on the split prefill schedule: the tiles of more
    than 64 pairs first, then the others, each part in tile order, i.e. a stable
    partition of the tile list (which the route tests check against the oracle); the
    first part's count in n_tiles[1].  multi_block_route: above 8192 pairs, where the
    order comes from the three-kernel route."""
    if case == "multi_block_route":
        # 8800 pairs over 64 experts, Zipf routing: heavy experts in several tiles, light ones
        cfg = LayerConfig("split_mb", 1100, 128, 128, 64, 8, seed=31, routing="zipf")
        li = make_inputs(cfg, "cpu").to("cuda")
    else:
        loads = SPLIT_LOADS if case == "mixed" else SPLIT_LOADS_WIDE
        flat = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(loads)])
        flat = flat[torch.randperm(flat.numel(), generator=torch.Generator().manual_seed(5))]
        M = flat.numel() // 2
        li = make_inputs(LayerConfig(f"order_{case}", M, 256, 128, len(loads), 2, seed=3), "cpu")
        li.topk_ids = flat[: M * 2].view(M, 2).contiguous()
        li = li.to("cuda")
    tiles, order, nwide = _tile_order_of(li, qmoe.QMOE_SCHED_PREFILL)
    wide = [t for t in range(len(tiles)) if tiles[t, 2] > 64]
    small = [t for t in range(len(tiles)) if tiles[t, 2] <= 64]
    assert nwide == len(wide)
    assert order.tolist() == wide + small
    assert len(small) > 0 or case == "all_wide"


def test_duplicate_experts_and_bad_ids():
    cfg = LayerConfig("dup", 24, 256, 128, 4, 3, seed=5)
    li = make_inputs(cfg, "cpu").to("cuda")
    ids = li.topk_ids.clone()
    ids[:, 1] = ids[:, 0]           # the same expert twice in a token
    ids[3, 2] = 9                   # >= E: skipped and flagged
    ids[5, 2] = -1
    li.topk_ids = ids.contiguous()
    out, layer = gpu_forward(li, qmoe.QMOE_SCHED_AUTO)
    rc, flags = qmoe.qmoe_read_error(layer._ws)
    assert rc == qmoe.QMOE_ERR_BAD_ID and flags & qmoe.QMOE_FLAG_BAD_ID
    # the oracle skips ids >= E as well
    check_layer(li, out, layer._ws, qmoe.QMOE_SCHED_AUTO, what="duplicates")


@pytest.mark.parametrize("cfg", CONFIGS[1:], ids=lambda c: c.name)
def test_full_config_sampled_tokens(cfg):
    """The benchmark's launch configuration on each full workload: 64 random tokens plus
    the tokens of the heaviest expert's tail tile, of the lightest experts and of the
    second MMA chain of wide tiles, against the unconditioned oracle (check_layer)."""
    li = make_inputs(cfg, "cuda")
    torch.cuda.synchronize()
    out, layer = gpu_forward(li, qmoe.QMOE_SCHED_AUTO)
    rc, flags = qmoe.qmoe_read_error(layer._ws)
    assert rc == 0 and flags == 0
    toks = forced_tokens(li, qmoe.QMOE_SCHED_AUTO, n_random=64, seed=cfg.seed)
    check_layer(li, out, layer._ws, qmoe.QMOE_SCHED_AUTO, tokens=toks, what=cfg.name)
    # deterministic: a second call is bitwise equal
    out2, _ = gpu_forward(li, qmoe.QMOE_SCHED_AUTO, layer)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_zero_tokens_is_a_noop():
    li = make_inputs(CONFIGS[0], "cpu").to("cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    x = torch.empty(0, li.cfg.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    w = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    out = layer(x, ids, w)
    assert out.shape == (0, li.cfg.H)


@pytest.mark.parametrize("cfg", [c for c in CONFIGS if c.name.startswith("prefill")],
                         ids=lambda c: c.name)
def test_prefill_pair_schedule_full_size(cfg):
    """The two-SM prefill GEMM on the full prefill workloads: run-to-run deterministic and
    within the tolerance of the oracle on the forced tokens.  (It accumulates each
    output on one chain in K order; the one-SM kernel splits narrow tiles over several
    chains, so the two agree to rounding, not bit for bit.)"""
    li = make_inputs(cfg, "cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    s = qmoe.QMOE_SCHED_PREFILL_PAIR
    outs = [layer(li.x, li.topk_ids, li.topk_weights, sched=s).clone() for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), \
        "two-SM schedule not deterministic"
    toks = forced_tokens(li, s, n_random=32, seed=cfg.seed)
    check_layer(li, outs[1], layer._ws, s, tokens=toks, what=f"{cfg.name} two-SM")


@pytest.mark.parametrize("cfg", [CONFIGS[1], CONFIGS[3]], ids=lambda c: c.name)
def test_forward_replays_from_a_cuda_graph(cfg):
    """The forward is stream work only (a memset and kernel launches, no host sync), so
    it captures into a CUDA graph; replays give the eager call's output bit for bit."""
    li = make_inputs(cfg, "cuda")
    layer = qmoe.NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    ref = layer(li.x, li.topk_ids, li.topk_weights).clone()
    torch.cuda.synchronize()
    out = torch.empty_like(ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer(li.x, li.topk_ids, li.topk_weights, out=out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(li.x, li.topk_ids, li.topk_weights, out=out)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    rc, flags = qmoe.qmoe_read_error(layer._ws)
    assert rc == 0 and flags == 0
