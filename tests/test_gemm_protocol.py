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


def simulate(*, NMW, SL, RS, DG, ACCB, KS, BIN, nb128, n_units, seed, plant=None):
    """One CTA running n_units units of nb128 weight blocks each.  Returns normally or
    raises ProtocolError (unsafe access) / RuntimeError (deadlock)."""
    rng = random.Random(seed)
    nks = -(-nb128 // KS)
    last_halves = nb128 - (nks - 1) * KS
    total = n_units * nks
    rfull = [Bar(1) for _ in range(RS)]
    rempty = [Bar(4) for _ in range(RS)]
    sfull = [Bar(5 if h == 0 else 4) for _ in range(SL) for h in range(KS)]
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
        return last_halves if (it % nks) == nks - 1 else KS

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

    def mma_warp(m):
        bg = m  # BIN: next step whose pair rows this warp copies

        def issue_b():
            nonlocal bg
            if bg >= total:
                return
            sl = bg % SL
            while not sempty[sl].done(((bg // SL) & 1) ^ 1):
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

        if BIN:
            yield from issue_b()
        it = 0
        for local in range(n_units):
            ab = local % ACCB
            while not acce[ab].done(((local // ACCB) & 1) ^ 1):
                yield False
            check(local < ACCB or drained[ab] >= local - ACCB,
                  f"accumulator {ab} written for unit {local} before unit {local - ACCB} was drained")
            ks0 = (m - it % NMW + NMW) % NMW
            for ks in range(ks0, nks, NMW):
                sit = it + ks
                sl, sph = sit % SL, (sit // SL) & 1
                while not sfull[sl * KS].done(sph):
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
                if KS == 2 and (ks != nks - 1 or last_halves == 2):
                    while not sfull[sl * KS + 1].done(sph):
                        yield False
                    check(all(v == sit for v in a_slot[sl][1]),
                          f"A slot {sl} block 1 not written for step {sit}")

                def done(sl=sl, sit=sit):  # the commit covers every earlier MMA
                    read_done[sl][0] = max(read_done[sl][0], sit)
                    read_done[sl][1] = sit
                later(sempty[sl], done)
                if BIN:
                    yield from issue_b()
                yield True
            it += nks

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
        for local in range(n_units):
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


@pytest.mark.parametrize("cfg", [DECODE, PREFILL_WIDE, PREFILL_NARROW],
                         ids=["decode", "prefill_wide", "prefill_narrow"])
@pytest.mark.parametrize("nb128", [1, 2, 3, 7, 16])
def test_protocol_is_safe_and_live(cfg, nb128):
    for seed in range(12):
        simulate(**cfg, nb128=nb128, n_units=5, seed=seed)


@pytest.mark.parametrize("plant,cfg", [("slab1_on_bempty0", PREFILL_WIDE),
                                       ("no_bfull1_wait", PREFILL_NARROW),
                                       ("no_sempty_wait", DECODE)])
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
