"""The CPU oracle against its pins, and planted mistakes against the pins.

Every mutant below is a copy of the oracle source with one plausible mistake
(a swapped nibble order, up and gate exchanged, a dropped factor, a wrong index,
a truncating rounding, an unstable sort...).  Each must fail at least one pin,
which shows that the pins constrain every step of the oracle.
"""

import os
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "qmoe_oracle.c")


@pytest.fixture(scope="module")
def lib():
    return oracle._load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


MUTANTS = {
    "nibble_order": ("(k & 1) ? (byte >> 4) : (byte & 0xF)", "(k & 1) ? (byte & 0xF) : (byte >> 4)"),
    "up_gate_swapped": ("double up = g[i], gate = g[I + i];", "double up = g[I + i], gate = g[i];"),
    "gscale13_dropped": ("g[n] = (double)gs13[e] * sum;", "g[n] = sum;"),
    "gscale2_dropped": ("double y = (double)gs2[e] * sum;", "double y = sum;"),
    "scale_block_index": ("s[n * (K / 16) + k / 16]", "s[n * (K / 16) + k / 32]"),
    "h_not_rounded": ("h[i] = qo_bf16_to_double(qo_bf16_rne(exact));", "h[i] = exact;"),
    "h_given_ignored": ("            h[i] = given;\n", "\n"),
    "h_bracket_one_sided": ("if (!(given >= lo && given <= hi)) n_out += 1;", "if (!(given >= lo)) n_out += 1;"),
    "h_bound_no_running_sum": ("err += fabs(slice) + fabs(sum);", "err += fabs(slice);"),
    "h_bound_worst_case_wide": ("ga[n] = fabs((double)gs13[e]) * 2.0 * u * err;",
                                "ga[n] = fabs((double)gs13[e]) * 2.0 * u * err * 200.0;"),
    "h_bound_first_order_only": ("1.1 * (fabs(up) + d_up) * d_gate", "1.1 * fabs(up) * d_gate"),
    "w4a4_e4m3_ties_up": ("double r = rint(v / q) * q;         /* nearest, ties to even */",
                          "double r = floor(v / q + 0.5) * q;"),
    "w4a4_e2m1_ties_odd": ("(d == bd && (c & 1) == 0 && (best & 1) == 1)", "(d == bd && (c & 1) == 1)"),
    "w4a4_global_scale": ("double g = amax / (6.0 * 448.0);\n  if (g == 0.0) g = 1.0;\n  for (int64_t b",
                          "double g = amax / 448.0;\n  if (g == 0.0) g = 1.0;\n  for (int64_t b"),
    "w4a4_h_not_quantized": ("        qo_nvfp4_row(h, I);\n", "\n"),
    "w4a4_x_not_quantized": ("      qo_nvfp4_row(xq, H);\n", "\n"),
    "h_flip_uncounted": ("if (given != h[i]) n_flip += 1;", ";"),
    "routing_weight_dropped": ("acc[j] += (double)topk_w[m * top_k + k] * y;", "acc[j] += y;"),
    "e2m1_sign_dropped": ("return (code & 8) ? -m : m;", "return m;"),
    "e2m1_table": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5}"),
    "e4m3_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "silu_sign": ("gate / (1.0 + exp(-gate))", "gate / (1.0 + exp(gate))"),
    "rounding_truncates": ("double r = rint(a / q) * q;", "double r = floor(a / q) * q;"),
    "x_row_ignored": ("qo_bf16_to_double(x[m * H + hh])", "qo_bf16_to_double(x[hh])"),
    "route_unstable": ("    int64_t pos = offsets[e] + seen[e];\n    seen[e] += 1;",
                       "    int64_t pos = offsets[e + 1] - 1 - seen[e];\n    seen[e] += 1;"),
    "tile_rows": ("if (rows > tile_n) rows = tile_n;", "if (rows >= tile_n) rows = tile_n - 1;"),
    "bad_id_counted": ("if (e >= 0 && e < E) count[e] += 1;", "if (e >= 0 && e < E) count[e] += 1; else if (e >= E) count[E-1] += 1;"),
    "limit_gate_ignored": ("if (gate > swiglu_limit) gate = swiglu_limit;", ";"),
    "limit_gate_two_sided": ("if (gate > swiglu_limit) gate = swiglu_limit;",
                             "if (gate > swiglu_limit) gate = swiglu_limit; if (gate < -swiglu_limit) gate = -swiglu_limit;"),
    "limit_up_one_sided": ("if (up < -swiglu_limit) up = -swiglu_limit;", ";"),
    "limit_after_silu": ("double silu = gate / (1.0 + exp(-gate));",
                         "double silu = g[I + i] / (1.0 + exp(-g[I + i]));"),
    "skip_negative_slot_wrong": ("        if (e < 0) continue;\n        if (e >= E) {", "        if (e < 0) e = 0;\n        if (e >= E) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "qmoe_oracle.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(d, "libmut.so")
        import subprocess
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so,
                        "-lm"], check=True)
        mut = oracle._load(so)
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(mut)
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"mutant {name} passed every pin"
