"""Model check of the grouped GEMM's mbarrier protocol (csrc/gemm.cu), on the CPU.

Every role of one CTA (weight producer, pair-row producer, MMA warps, dequant warps,
epilogue warps) runs as a coroutine that follows the kernel's waits and arrivals for
each schedule's configuration; asynchronous completions (TMA bytes landing,
tcgen05.commit arrivals) are delivered after random delays, in any order.  An mbarrier
is modelled by its count of completed phases: a parity wait passes when the latest
completed phase has that parity (a fresh barrier counts as having completed a phase
of parity 1), which is exactly what lets a role run a whole ring cycle ahead and pass
a wait early; the kernel's rule that every use of a slot or stage falls to one dequant
group and one MMA warp is what prevents that.

Checked for every seed: no deadlock, and data safety, i.e. no weight stage, A slot,
pair-row slab or accumulator is written while a reader of its previous contents may
still need it, and none is read before it holds its own step's data.  A planted
mistake (a slab refilled on the wrong barrier, a missing wait) must be caught.
"""

import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pend, self.completed = count, count, 0

    def expect_tx(self):
        self.pend += 1  # outstanding bytes count as one more arrival

    def arrive(self):
        self.pend -= 1
        assert self.pend >= 0, "over-arrival"
        if self.pend == 0:
            self.completed += 1
            self.pend = self.count

    def done(self, parity):
        return ((self.completed - 1) & 1) == parity


class ProtocolError(AssertionError):
    pass


def check(cond, msg):
    if not cond:
        raise ProtocolError(msg)


def segments(g0, total, nks):
    """Stream-K (BIN): the (unit, first step, steps) pieces of the global steps
    [g0, g0 + total), as the kernel's MMA and epilogue loops cut them."""
    out, it = [], 0
    while it < total:
        g = g0 + it
        u, k0 = divmod(g, nks)
        n = min(nks - k0, total - it)
        out.append((u, k0, n))
        it += n
    return out


def simulate(*, NMW, SL, RS, DG, ACCB, KS, BIN, nb128, n_units, seed, plant=None, g0=0, PB=False):
    """One CTA running n_units units of nb128 weight blocks each (BIN: the global steps
    [g0, g0 + n_units * nks) of the stream-K sequence, which may start and end inside
    a unit).  Returns normally or raises ProtocolError (unsafe access) / RuntimeError
    (deadlock)."""
    rng = random.Random(seed)
    nks = -(-nb128 // KS)
    last_halves = nb128 - (nks - 1) * KS
    total = n_units * nks
    segs = segments(g0, total, nks) if BIN else [(u, 0, nks) for u in range(n_units)]
    rfull = [Bar(1) for _ in range(RS)]
    rempty = [Bar(4) for _ in range(RS)]
    # PB: the decode pipeline with a pair-row producer warp; the copy counts on the step's
    # last block barrier, and the MMA warps wait on that one alone
    lastb = KS - 1 if PB else 0
    sfull = [Bar(5 if h == lastb else 4) for _ in range(SL) for h in range(KS)]
    sempty = [Bar(1) for _ in range(SL)]
    bempty0 = [Bar(1) for _ in range(SL)]
    bfull1 = [Bar(1) for _ in range(SL)]
    accf = [Bar(NMW) for _ in range(ACCB)]
    acce = [Bar(4) for _ in range(ACCB)]
    pending = []  # [delay, barrier, effect]

    def later(bar, effect=None, hi=25):
        pending.append([rng.randint(1, hi), bar, effect])

    # data state
    raw = [-1] * RS                                  # step a weight stage holds
    a_slot = [[[-1] * 4 for _ in range(KS)] for _ in range(SL)]  # [slot][block][quarter]
    b_slab = [[-1, -1] for _ in range(SL)]           # step whose pair rows a slab holds
    read_done = [[-1, -1] for _ in range(SL)]        # last step whose MMAs of slab h completed
    unit_mma_done = [[-1] * NMW for _ in range(ACCB)]  # last unit whose MMAs (warp m) completed
    drained = [-1] * ACCB                            # last unit the epilogue finished
    drained_by = [[-1] * 4 for _ in range(ACCB)]

    def step_blocks(it):
        return last_halves if ((g0 + it) % nks) == nks - 1 else KS

    def weight_producer():
        for it in range(total):
            s = it % RS
            while not rempty[s].done(((it // RS) & 1) ^ 1):
                yield False
            rfull[s].expect_tx()
            rfull[s].arrive()

            def land(s=s, it=it):
                raw[s] = it
            later(rfull[s], land)
            yield True

    def pair_producer():  # 2-D boxes, slab by slab (prefill)
        for it in range(total):
            s, eph = it % SL, ((it // SL) & 1) ^ 1
            for sl in range(2):
                eb = bempty0[s] if sl == 0 else sempty[s]
                if plant == "slab1_on_bempty0":
                    eb = bempty0[s]
                while not eb.done(eph):
                    yield False
                check(it < SL or read_done[s][sl] >= it - SL,
                      f"slab {s}.{sl} refilled for step {it} while step {it - SL} may read it")
                fb = sfull[s * KS] if sl == 0 else bfull1[s]
                fb.expect_tx()
                fb.arrive()

                def land(s=s, sl=sl, it=it):
                    b_slab[s][sl] = it
                later(fb, land)
                yield True

    def pair_producer_bin():  # PB: the producer warp, up to SL steps ahead
        for bg in range(total):
            sl = bg % SL
            while plant != "no_b_wait" and not sempty[sl].done(((bg // SL) & 1) ^ 1):
                yield False
            check(bg < SL or read_done[sl][0] >= bg - SL,
                  f"pair rows of slot {sl} refilled for step {bg} too early")
            fb = sfull[sl * KS + lastb]
            fb.expect_tx()
            fb.arrive()

            def land(sl=sl, g=bg):
                b_slab[sl][0] = b_slab[sl][1] = g
            later(fb, land)
            yield True

    def mma_warp(m):
        bg = m  # BIN: next step whose pair rows this warp copies

        def issue_b():
            nonlocal bg
            if bg >= total:
                return
            sl = bg % SL
            while plant != "no_b_wait" and not sempty[sl].done(((bg // SL) & 1) ^ 1):
                yield False
            check(bg < SL or read_done[sl][0] >= bg - SL,
                  f"pair rows of slot {sl} refilled for step {bg} too early")
            fb = sfull[sl * KS]
            fb.expect_tx()
            fb.arrive()

            def land(sl=sl, g=bg):
                b_slab[sl][0] = b_slab[sl][1] = g
            later(fb, land)
            bg += NMW

        if BIN and not PB:
            yield from issue_b()
        it = 0
        for local, (_, k0, seg_len) in enumerate(segs):
            ab = local % ACCB
            while not acce[ab].done(((local // ACCB) & 1) ^ 1):
                yield False
            check(local < ACCB or drained[ab] >= local - ACCB,
                  f"accumulator {ab} written for unit {local} before unit {local - ACCB} was drained")
            ks0 = (m - it % NMW + NMW) % NMW
            for ks in range(ks0, seg_len, NMW):
                sit = it + ks
                sl, sph = sit % SL, (sit // SL) & 1
                while not sfull[sl * KS + lastb].done(sph):
                    yield False
                check(all(v == sit for v in a_slot[sl][0]), f"A slot {sl} not written for step {sit}")
                check(b_slab[sl][0] == sit, f"pair rows of slot {sl} not landed for step {sit}")
                if not BIN:
                    def done0(sl=sl, sit=sit):
                        read_done[sl][0] = max(read_done[sl][0], sit)
                    later(bempty0[sl], done0)
                    if plant != "no_bfull1_wait":
                        while not bfull1[sl].done(sph):
                            yield False
                    check(b_slab[sl][1] == sit, f"slab {sl}.1 not landed for step {sit}")
                if KS == 2 and (k0 + ks != nks - 1 or last_halves == 2):
                    while not PB and not sfull[sl * KS + 1].done(sph):
                        yield False
                    check(all(v == sit for v in a_slot[sl][1]),
                          f"A slot {sl} block 1 not written for step {sit}")

                def done(sl=sl, sit=sit):  # the commit covers every earlier MMA
                    read_done[sl][0] = max(read_done[sl][0], sit)
                    read_done[sl][1] = sit
                later(sempty[sl], done)
                if BIN and not PB:
                    yield from issue_b()
                yield True
            it += seg_len

            def unit_done(ab=ab, local=local):
                unit_mma_done[ab][m] = local
            later(accf[ab], unit_done)
            yield True

    def dequant_warp(g, q):
        for it in range(g, total, DG):
            s, a = it % RS, it % SL
            while not rfull[s].done((it // RS) & 1):
                yield False
            check(raw[s] == it, f"weight stage {s} holds step {raw[s]}, not {it}")
            rempty[s].arrive()
            if plant != "no_sempty_wait":
                while not sempty[a].done(((it // SL) & 1) ^ 1):
                    yield False
            check(it < SL or read_done[a][1] >= it - SL,
                  f"A slot {a} rewritten for step {it} while step {it - SL} may read it")
            for h in range(KS):
                if h < step_blocks(it):
                    a_slot[a][h][q] = it
                sfull[a * KS + h].arrive()
            yield True

    def epilogue_warp(q):
        for local in range(len(segs)):
            ab = local % ACCB
            while not accf[ab].done((local // ACCB) & 1):
                yield False
            check(all(v == local for v in unit_mma_done[ab]),
                  f"unit {local} read before all its MMAs completed")
            drained_by[ab][q] = local
            if all(v == local for v in drained_by[ab]):
                drained[ab] = local
            acce[ab].arrive()
            yield True

    roles = [weight_producer()]
    if not BIN:
        roles.append(pair_producer())
    elif PB:
        roles.append(pair_producer_bin())
    roles += [mma_warp(m) for m in range(NMW)]
    roles += [dequant_warp(g, q) for g in range(DG) for q in range(4)]
    roles += [epilogue_warp(q) for q in range(4)]
    idle = 0
    while roles:
        progress = False
        for p in pending:
            p[0] -= 1
        for p in [p for p in pending if p[0] <= 0]:
            pending.remove(p)
            if p[2]:
                p[2]()
            p[1].arrive()
            progress = True
        rng.shuffle(roles)
        for r in list(roles):
            try:
                progress |= next(r)
            except StopIteration:
                roles.remove(r)
                progress = True
        idle = 0 if (progress or pending) else idle + 1
        if idle > 3:
            raise RuntimeError("deadlock")


# the kernel's launch configurations (launch_gemm in csrc/gemm.cu)
DECODE = dict(NMW=3, SL=3, RS=9, DG=3, ACCB=2, KS=2, BIN=True)
PREFILL_WIDE = dict(NMW=1, SL=2, RS=6, DG=2, ACCB=1, KS=1, BIN=False)
PREFILL_NARROW = dict(NMW=1, SL=2, RS=8, DG=2, ACCB=2, KS=1, BIN=False)
# the split prefill schedule's small tiles: the decode pipeline with one MMA warp
PREFILL_SMALL = dict(NMW=2, SL=2, RS=8, DG=2, ACCB=2, KS=2, BIN=True, PB=True)
PREFILL_SMALL_1MMA = dict(NMW=1, SL=3, RS=6, DG=3, ACCB=2, KS=2, BIN=True, PB=True)


@pytest.mark.parametrize("cfg", [DECODE, PREFILL_WIDE, PREFILL_NARROW, PREFILL_SMALL,
                                 PREFILL_SMALL_1MMA],
                         ids=["decode", "prefill_wide", "prefill_narrow", "prefill_small",
                              "prefill_small_1mma"])
@pytest.mark.parametrize("nb128", [1, 2, 3, 7, 16])
def test_protocol_is_safe_and_live(cfg, nb128):
    for seed in range(12):
        simulate(**cfg, nb128=nb128, n_units=5, seed=seed)


@pytest.mark.parametrize("nb128,g0", [(7, 5), (16, 3), (16, 15), (3, 1), (2, 0)])
def test_stream_k_ranges_are_safe_and_live(nb128, g0):
    """The decode schedule's CTAs start and end inside units (stream-K)."""
    for seed in range(12):
        simulate(**DECODE, nb128=nb128, n_units=4, seed=seed, g0=g0)


def _range_start(n_steps, c, G):
    return n_steps * c // G


def _cta_of(g, n_steps, G):
    return ((g + 1) * G + n_steps - 1) // n_steps - 1


def _split(n_units, nks, G):
    waves = (n_units + G - 1) // G
    return (waves * G - n_units) * nks > 2 * G


def test_stream_k_split_rule():
    """Units are split between CTAs only where whole units would leave more than two K
    steps per CTA idle on average: the decode workloads' FC1 (384 units of 28 steps,
    3300 of 28) split, their FC2 (448 of 12, 5600 of 8) do not."""
    assert _split(384, 28, 152) and _split(3300, 28, 152)
    assert not _split(448, 12, 152) and not _split(5600, 8, 152)
    assert not _split(152, 28, 152) and _split(153, 28, 152) and _split(1, 28, 152)
    assert not _split(1, 1, 152)


@pytest.mark.parametrize("n_units,G", [(448, 152), (5600, 152), (7, 3), (1, 1)])
def test_whole_unit_ranges(n_units, G):
    """Without splitting, CTA c takes units [n_units c / G, n_units (c + 1) / G): every unit
    once, at most ceil(n_units / G) per CTA, no partial pieces."""
    nks = 5
    seen = []
    for c in range(G):
        u0, u1 = _range_start(n_units, c, G), _range_start(n_units, c + 1, G)
        assert u1 - u0 <= -(-n_units // G)
        for u, k0, n in segments(u0 * nks, (u1 - u0) * nks, nks):
            assert k0 == 0 and n == nks
            seen.append(u)
    assert seen == list(range(n_units))


@pytest.mark.parametrize("n_units,nks,G", [(384, 28, 152), (3200, 28, 152), (448, 12, 152),
                                           (1, 28, 152), (3, 4, 152), (5, 1, 7), (152, 1, 152),
                                           (153, 2, 152), (7, 28, 10), (1, 1, 1)])
def test_stream_k_partition_and_reduction(n_units, nks, G):
    """The formulas of the decode schedule's stream-K split (sk_range_start, sk_cta_of and
    the partial slots of sk_reduce in csrc/gemm.cu), over all CTAs: every step is in
    exactly one range; a unit's pieces lie in the CTAs sk_cta_of names, in K order; the
    pieces counted by the reduction are the real ones; no CTA writes two partials into
    one slot, and the reducer reads each CTA's partial from the slot it was written to;
    no two split units share an arrival counter (indexed by the unit's first CTA)."""
    T = n_units * nks
    starts = [_range_start(T, c, G) for c in range(G + 1)]
    assert starts[0] == 0 and starts[G] == T
    owner = {}
    written = {}  # (cta, slot) -> unit
    pieces = {u: [] for u in range(n_units)}
    for c in range(G):
        g0, total = starts[c], starts[c + 1] - starts[c]
        for u, k0, n in segments(g0, total, nks):
            for k in range(k0, k0 + n):
                assert (u, k) not in owner
                owner[(u, k)] = c
            pieces[u].append((c, k0, n))
            if not (k0 == 0 and n == nks):          # a partial: sk_reduce stores it
                slot = 0 if g0 // nks == u else 1
                assert (c, slot) not in written, "two partials in one slot"
                written[(c, slot)] = u
    assert len(owner) == T
    counter_of = {}  # the reduction's counter index: the CTA holding the unit's first step
    for u, ps in pieces.items():
        c0, c1 = _cta_of(u * nks, T, G), _cta_of(u * nks + nks - 1, T, G)
        if len(ps) > 1:
            assert c0 not in counter_of, "two split units share an arrival counter"
            counter_of[c0] = u
        real = [c for c, _, _ in ps]
        counted = [c for c in range(c0, c1 + 1) if starts[c + 1] > starts[c]]
        assert counted == real == sorted(real)
        assert [k0 for _, k0, _ in ps] == sorted(k0 for _, k0, _ in ps)
        if len(ps) > 1:
            for c in real:
                slot = 0 if starts[c] // nks == u else 1
                assert written[(c, slot)] == u


@pytest.mark.parametrize("plant,cfg", [("slab1_on_bempty0", PREFILL_WIDE),
                                       ("no_bfull1_wait", PREFILL_NARROW),
                                       ("no_sempty_wait", DECODE),
                                       ("no_sempty_wait", PREFILL_SMALL),
                                       ("no_b_wait", PREFILL_SMALL),
                                       ("no_b_wait", DECODE)])
def test_planted_protocol_mistakes_are_caught(plant, cfg):
    with pytest.raises((ProtocolError, RuntimeError)):
        for seed in range(30):
            simulate(**cfg, nb128=7, n_units=5, seed=seed, plant=plant)


def test_parity_aliasing_rule_is_needed():
    """Slots that do not all fall to one dequant group (SL % DG != 0) let a group pass
    a slot's wait a full ring cycle early: the model must fail on some seed."""
    bad = dict(DECODE, SL=4)  # 4 slots, 3 dequant groups and 3 MMA warps
    with pytest.raises((ProtocolError, RuntimeError)):
        for seed in range(60):
            simulate(**bad, nb128=16, n_units=6, seed=seed)
