"""GPU parity at the edges of the accepted shapes, against the CPU oracle: the largest
expert count and top_k the ABI takes, the smallest H and I, a single token with a
single slot, and a batch just above the size where the route switches to its
multi-block form.  Same checks as tests/test_gpu_forward.py."""

import numpy as np
import pytest
import torch

from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import LayerConfig, make_inputs
from tests.helpers import check_layer, gpu_forward

pytestmark = pytest.mark.gpu

EDGES = [
    # name, M, H, I, E, top_k, experts drawn (None: all E)
    ("max_E_max_topk", 70, 256, 128, 2048, 64, 200),
    ("min_H_I", 33, 128, 128, 4, 2, None),
    ("one_token_one_slot", 1, 256, 256, 3, 1, None),
    ("route_multi_block", 4097, 128, 128, 8, 2, None),
]


def _inputs(name, M, H, I, E, k, n_draw):
    cfg = LayerConfig(name, M, H, I, E, k, seed=41)
    if n_draw is None:
        return make_inputs(cfg, "cpu").to("cuda")
    # many experts: route the tokens to a random subset so that only those experts'
    # weights need drawing (the others stay zero and are never touched)
    rng = np.random.default_rng(7)
    experts = rng.choice(E, size=n_draw, replace=False)
    li = make_inputs(cfg, "cpu", experts=experts)
    ids = np.stack([rng.choice(experts, size=k, replace=False) for _ in range(M)])
    li.topk_ids = torch.from_numpy(ids.astype(np.int32))
    w = rng.random((M, k)).astype(np.float32)
    li.topk_weights = torch.from_numpy(w / w.sum(1, keepdims=True))
    return li.to("cuda")


@pytest.mark.parametrize("edge", EDGES, ids=lambda e: e[0])
@pytest.mark.parametrize("sched", [qmoe.QMOE_SCHED_AUTO, qmoe.QMOE_SCHED_DECODE,
                                   qmoe.QMOE_SCHED_PREFILL])
def test_edge_shape(edge, sched):
    name, M, H, I, E, k, n_draw = edge
    li = _inputs(name, M, H, I, E, k, n_draw)
    out, layer = gpu_forward(li, sched)
    rc, flags = qmoe.qmoe_read_error(layer._ws)
    assert rc == 0 and flags == 0
    toks = None
    if M > 64:
        rng = np.random.default_rng(M)
        toks = np.unique(np.concatenate([[0, M - 1], rng.choice(M, 30, replace=False)]))
    check_layer(li, out, layer._ws, sched, tokens=toks, what=f"{name} sched={sched}")
