"""The oracle's h-acceptance bound at production size (H = 7168), on the CPU.

The GPU parity tests accept a GPU bf16 h value that differs from the oracle's own
rounding only if it is the bf16 rounding of some value within delta of the exact
SiLU(gate)*up; delta is the first-order error of an fp32 accumulation of 16-wide slice
sums (the oracle's header states it).  Here the bound meets an emulation of the
grouped GEMM's arithmetic (tests/oracle_pins.emulate_fc1_h) on 64 tokens x 512
intermediate values of random NVFP4 rows with H = 7168:

  * every emulated h (one accumulator as on the prefill schedules or three as on the
    decode schedule; each rounding to nearest or, least favourably, toward zero) must
    be accepted;
  * a value two bf16 steps from the oracle's own rounding must be rejected, except
    where the exact value's own bound reaches past the neighbouring bf16 value
    (cancelling dot products), at most 2% of the values (about 1.1% here);
  * the emulated share of h values rounded the other way (flips) must stay under
    MAX_FLIP_RATE, the limit the GPU parity tests apply.
"""

import pytest

from tests import oracle_pins
from tests.helpers import MAX_FLIP_RATE

import oracle

M, I = 64, 512


@pytest.fixture(scope="module")
def layer():
    li, x, w13, gs = oracle_pins.h_bound_layer(M, I)
    own = oracle.forward(li.x, li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2, li.topk_ids,
                         li.topk_weights, return_h=True)[1]["h"]
    return li, x, w13, gs, own


@pytest.mark.parametrize("chains,truncate", [(1, False), (3, False), (1, True), (3, True)],
                         ids=["one_chain_rne", "three_chains_rne", "one_chain_trunc",
                              "three_chains_trunc"])
def test_emulated_fp32_accumulation_is_accepted(layer, chains, truncate):
    li, x, w13, gs, _ = layer
    hg = oracle_pins.emulate_fc1_h(x, w13, gs, chains, truncate)
    st = oracle_pins.h_given_stats(oracle._load(), li, hg)
    assert st["compared"] == M * I
    assert st["outside"] == 0, f"{st['outside']} emulated fp32 roundings rejected by the bound"
    rate = st["flipped"] / st["compared"]
    print(f"[h-bound] chains={chains} truncate={truncate}: {st['flipped']} of {st['compared']} "
          f"h values rounded the other way ({rate:.2e})")
    assert rate <= MAX_FLIP_RATE
    # fp32 accumulation at this size must flip some roundings, or the emulation is not
    # exercising the bound at all
    assert st["flipped"] > 0


@pytest.mark.parametrize("direction", [+2, -2], ids=["two_steps_out", "two_steps_in"])
def test_two_steps_away_is_rejected(layer, direction):
    li, _, _, _, own = layer
    far, moved = oracle_pins.two_steps_away(own, direction)
    st = oracle_pins.h_given_stats(oracle._load(), li, far)
    accepted = moved - st["outside"]
    print(f"[h-bound] {direction:+d} steps: {accepted} of {moved} moved values still accepted")
    assert accepted <= 0.02 * moved
