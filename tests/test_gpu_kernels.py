"""GPU parity of the building blocks: dequant, repack layout, route tables, errors.

All calls go through the C-ABI (libqmoe.so) via the ctypes binding.
"""

import zlib

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_grouped_route_gb300 import qmoe
from qmoe_inputs import CONFIGS
from qmoe_inputs.gen import _routing

pytestmark = pytest.mark.gpu


def test_dequant_every_code_and_scale():
    """kernel dequant(code, scale) == E2M1(code) * E4M3(scale), all 16 x 256 pairs at
    each of the 8 element positions of a packed word (the other positions holding other
    codes), exact."""
    got = qmoe.qmoe_selftest_dequant().cpu().numpy().astype(np.uint16).reshape(16, 256, 8)
    gotf = oracle.bf16_bits_to_float(got)
    for c in range(16):
        for j in range(8):
            code = (c + j) % 16
            for s in range(256):
                want = oracle.dec_e2m1(code) * oracle.dec_e4m3(s)
                if np.isnan(want):
                    assert np.isnan(gotf[c, s, j]), (c, j, s)
                else:
                    assert gotf[c, s, j] == want, (c, j, s, gotf[c, s, j], want)


def _unpack_repacked(codes: np.ndarray, scales: np.ndarray, E, N, K, w13: bool):
    """Invert the documented repack layout on the CPU -> plain codes [E][N][K] and
    scales [E][N][K/16]."""
    nrb, nks = N // 128, K // 128
    words = codes.view(np.uint32).reshape(E, nrb, nks, 4, 128, 4)
    # element j of a packed word -> (bit positions of magnitude bits 0,1,2 and sign)
    pos = {0: (6, 7, 8, 15), 1: (22, 23, 24, 31), 2: (0, 1, 2, 9), 3: (16, 17, 18, 25),
           4: (26, 27, 28, 3), 5: (10, 11, 12, 19), 6: (4, 5, 14, 13), 7: (20, 21, 30, 29)}
    plain = np.zeros((E, nrb, nks, 4, 128, 4, 8), np.uint8)
    for j, (b0, b1, b2, bs) in pos.items():
        v = (((words >> b0) & 1) | (((words >> b1) & 1) << 1) | (((words >> b2) & 1) << 2)
             | (((words >> bs) & 1) << 3))
        plain[..., j] = v.astype(np.uint8)
    # -> [E][nrb][128 rows][nks][kk][wd][8] = K order within the row
    plain = plain.transpose(0, 1, 4, 2, 3, 5, 6).reshape(E, nrb, 128, K)
    sc = scales.reshape(E, nrb, nks, 128, 8).transpose(0, 1, 3, 2, 4).reshape(E, nrb, 128, K // 16)
    out_c = np.zeros((E, N, K), np.uint8)
    out_s = np.zeros((E, N, K // 16), np.uint8)
    I = N // 2
    for rb in range(nrb):
        for r in range(128):
            if w13:
                q, j = r >> 5, r & 31
                i = rb * 64 + q * 16 + (j & 15)
                n = i if j < 16 else I + i
            else:
                n = rb * 128 + r
            out_c[:, n] = plain[:, rb, r]
            out_s[:, n] = sc[:, rb, r]
    return out_c, out_s


@pytest.mark.parametrize("which", [qmoe.QMOE_W13, qmoe.QMOE_W2])
def test_repack_is_the_documented_permutation(which):
    g = torch.Generator(device="cuda").manual_seed(3)
    E, N, K = 3, 384, 256
    w = torch.randint(0, 256, (E, N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
    s = torch.randint(0, 256, (E, N, K // 16), dtype=torch.uint8, device="cuda", generator=g)
    codes, scales = qmoe.moe_nvfp4_repack(w, s, which)
    torch.cuda.synchronize()
    pc, ps = _unpack_repacked(codes.cpu().numpy(), scales.cpu().numpy(), E, N, K,
                              which == qmoe.QMOE_W13)
    wn = w.cpu().numpy()
    want_codes = np.stack([wn & 0xF, wn >> 4], axis=-1).reshape(E, N, K)
    assert np.array_equal(pc, want_codes)
    assert np.array_equal(ps, s.cpu().numpy())


def _check_route(ids: torch.Tensor, E: int, tile_n: int):
    offsets, sp, pp, tiles, n_tiles, ws = qmoe.moe_route(ids, E, tile_n)
    torch.cuda.synchronize()
    o_off, o_sp, o_pp, o_tiles, rc = oracle.route(ids.cpu().numpy(), E, tile_n)
    assert np.array_equal(offsets.cpu().numpy(), o_off)
    assert np.array_equal(sp.cpu().numpy(), o_sp)
    assert np.array_equal(pp.cpu().numpy(), o_pp)
    nt = int(n_tiles.item())
    assert nt == o_tiles.shape[0]
    assert np.array_equal(tiles[:nt].cpu().numpy(), o_tiles)
    flags_rc, flags = qmoe.qmoe_read_error(ws)
    assert bool(flags & qmoe.QMOE_FLAG_BAD_ID) == (rc == oracle.QO_WARN_BAD_ID)


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: c.name)
@pytest.mark.parametrize("tile_n", [16, 32, 256, 320])
def test_route_configs_bit_exact(cfg, tile_n):
    g = torch.Generator(device="cuda").manual_seed(cfg.seed)
    ids, _ = _routing(cfg, g, "cuda")
    _check_route(ids.contiguous(), cfg.E, tile_n)


@pytest.mark.parametrize("case", ["neg_ids", "bad_ids", "one_expert", "all_same", "empty_experts",
                                  "nothing_routed", "tile1", "big_E", "ragged",
                                  # above 8192 pairs: the three-kernel multi-block route
                                  "mb_bad_ids", "mb_big_E", "mb_one_expert", "mb_just_above",
                                  "mb_nothing_routed"])
def test_route_edge_cases(case):
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    if case == "neg_ids":
        ids, E, T = rng.integers(-1, 6, size=(97, 3)), 6, 16
    elif case == "bad_ids":
        ids, E, T = rng.integers(-2, 9, size=(50, 4)), 7, 32
    elif case == "one_expert":
        ids, E, T = np.zeros((33, 2)), 1, 16
    elif case == "all_same":
        ids, E, T = np.full((700, 8), 5), 8, 256
    elif case == "empty_experts":
        ids, E, T = rng.choice([3, 77, 200], size=(64, 8)), 256, 32
    elif case == "nothing_routed":
        ids, E, T = np.full((9, 4), -1), 16, 32
    elif case == "tile1":
        ids, E, T = rng.integers(0, 5, size=(20, 3)), 5, 1
    elif case == "big_E":
        ids, E, T = rng.integers(0, 2048, size=(1000, 8)), 2048, 256
    elif case == "ragged":
        ids, E, T = rng.integers(0, 3, size=(1001, 1)), 3, 256
    elif case == "mb_bad_ids":
        ids, E, T = rng.integers(-2, 12, size=(3001, 3)), 10, 320
    elif case == "mb_big_E":
        ids, E, T = rng.integers(0, 2048, size=(2500, 8)), 2048, 192
    elif case == "mb_one_expert":
        ids, E, T = np.zeros((10000, 1)), 1, 320
    elif case == "mb_just_above":
        ids, E, T = rng.integers(0, 3, size=(8193, 1)), 3, 16
    else:
        ids, E, T = np.full((4097, 4), -1), 16, 320
    _check_route(torch.tensor(np.asarray(ids), dtype=torch.int32, device="cuda"), E, T)


def test_route_large_prefill_distribution():
    g = torch.Generator(device="cuda").manual_seed(99)
    ids = torch.randint(-1, 256, (8192, 8), generator=g, device="cuda", dtype=torch.int32)
    _check_route(ids, 256, 256)


def test_timeout_is_reported_not_hung():
    rc = qmoe.qmoe_selftest_timeout(2_000_000)  # 2 ms
    assert rc == qmoe.QMOE_ERR_TIMEOUT
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


def test_error_word_bits_map_to_return_codes():
    """qmoe_read_error: the internal-check bit wins over timeout, timeout over bad id."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for word, want in [(0, qmoe.QMOE_OK), (qmoe.QMOE_FLAG_BAD_ID, qmoe.QMOE_ERR_BAD_ID),
                       (qmoe.QMOE_FLAG_TIMEOUT | qmoe.QMOE_FLAG_BAD_ID, qmoe.QMOE_ERR_TIMEOUT),
                       (qmoe.QMOE_FLAG_INTERNAL | qmoe.QMOE_FLAG_TIMEOUT, qmoe.QMOE_ERR_CUDA)]:
        ws[:4] = torch.tensor([word], dtype=torch.int32).view(torch.uint8).to("cuda")
        rc, flags = qmoe.qmoe_read_error(ws)
        assert (rc, flags) == (want, word)


def test_argument_errors():
    x = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(4, 2, dtype=torch.int32, device="cuda")
    w = torch.zeros(1, dtype=torch.float32, device="cuda")
    u8 = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmoe.QmoeError) as ei:
        qmoe.moe_nvfp4_forward(x, u8, u8, w, u8, u8, w, ids, w.expand(4, 2).contiguous(),
                               H=100, I=128, E=1)
    assert ei.value.code == qmoe.QMOE_ERR_SHAPE
    with pytest.raises(qmoe.QmoeError) as ei:
        qmoe.moe_nvfp4_repack(torch.zeros(1, 100, 64, dtype=torch.uint8, device="cuda"),
                              torch.zeros(1, 100, 8, dtype=torch.uint8, device="cuda"), qmoe.QMOE_W2)
    assert ei.value.code == qmoe.QMOE_ERR_SHAPE
