"""Property tests of the CPU oracle's route and of the scale layout, on random inputs
drawn by hypothesis (skipped where hypothesis is not installed)."""

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import scale_layout  # noqa: E402


@settings(max_examples=60, deadline=None)
@given(M=st.integers(0, 40), k=st.integers(1, 6), E=st.integers(1, 12), T=st.integers(1, 40),
       seed=st.integers(0, 2**31 - 1))
def test_route_is_the_stable_sort(M, k, E, T, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-2, E + 2, size=(M, k)).astype(np.int32)
    off, sp, pp, tiles, rc = oracle.route(ids, E, T)
    flat = ids.reshape(-1)
    valid = [i for i in range(flat.size) if 0 <= flat[i] < E]
    order = sorted(valid, key=lambda i: (flat[i], i))
    assert list(sp[:len(order)]) == order and all(v == -1 for v in sp[len(order):])
    for pos, i in enumerate(order):
        assert pp[i] == pos
    assert all(pp[i] == -1 for i in range(flat.size) if not 0 <= flat[i] < E)
    counts = np.bincount([flat[i] for i in valid], minlength=E) if valid else np.zeros(E, int)
    assert list(off) == [0] + list(np.cumsum(counts))
    # tiles: each expert's run cut into pieces of at most T, in order, covering it once
    want = [(e, off[e] + s, min(T, counts[e] - s)) for e in range(E) for s in range(0, counts[e], T)]
    assert [tuple(t) for t in tiles] == want
    assert (rc == oracle.QO_WARN_BAD_ID) == bool(((flat >= E)).any())


@settings(max_examples=40, deadline=None)
@given(nt=st.integers(1, 4), nu=st.integers(1, 6), E=st.integers(1, 3),
       seed=st.integers(0, 2**31 - 1))
def test_scale_layout_round_trips(nt, nu, E, seed):
    N, C = 128 * nt, 4 * nu
    rng = np.random.default_rng(seed)
    plain = rng.integers(0, 256, size=(E, N, C), dtype=np.uint8)
    swz = scale_layout.swizzle_128x4(plain)
    assert np.array_equal(scale_layout.unswizzle_128x4(swz, N, C), plain)
    assert np.array_equal(np.sort(swz, axis=1), np.sort(plain.reshape(E, -1), axis=1))
