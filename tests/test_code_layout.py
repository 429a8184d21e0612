"""The packed E2M1 code layout the repack writes and the GEMM's dequant reads, checked on
the CPU as a specification: for every code at every element position of a 32-bit word,
the documented shifts, rotation and masks put that code's magnitude bits on the bf16
mantissa/exponent positions 6-8 (22-24) and its sign on bit 15 (31) of the right output
half, and nothing else there.  The GPU tests check the kernels themselves
(test_gpu_kernels: every code and scale at every position through the device dequant,
and the repacked bytes against this bit table).
"""

import pytest

M = 0x81C081C0
MASK32 = 0xFFFFFFFF

# element j -> positions in the packed word of its magnitude bits 0, 1, 2 and sign
POS = {0: (6, 7, 8, 15), 1: (22, 23, 24, 31), 2: (0, 1, 2, 9), 3: (16, 17, 18, 25),
       4: (26, 27, 28, 3), 5: (10, 11, 12, 19), 6: (4, 5, 14, 13), 7: (20, 21, 30, 29)}


def pack(codes):
    q = 0
    for j, c in enumerate(codes):
        b0, b1, b2, bs = POS[j]
        q |= (c & 1) << b0 | ((c >> 1) & 1) << b1 | ((c >> 2) & 1) << b2 | ((c >> 3) & 1) << bs
    return q


def outputs(q):
    """The four bf16x2 words before the scale multiply, as the dequant forms them."""
    rot12 = ((q << 12) | (q >> 20)) & MASK32
    return [q & M,
            (q << 6) & M & MASK32,
            rot12 & M,
            (((q << 2) & 0x80C080C0) | ((q >> 6) & 0x01000100)) & MASK32]


def placed(code):
    """code s|e1 e0 m as bf16 bits: magnitude at 6-8, sign at 15 (code * 2^-126)."""
    return ((code >> 3) & 1) << 15 | (code & 7) << 6


def test_every_bit_of_the_word_holds_one_code_bit():
    bits = [b for j in range(8) for b in POS[j]]
    assert sorted(bits) == list(range(32))


@pytest.mark.parametrize("j", range(8))
def test_each_position_reaches_its_output_half(j):
    for code in range(16):
        for other in (0, 5, 15):
            codes = [other] * 8
            codes[j] = code
            out = outputs(pack(codes))
            half = (out[j // 2] >> (16 * (j % 2))) & 0xFFFF
            assert half == placed(code), (j, code, other, hex(half))


def test_placed_bits_are_the_e2m1_value_times_2_to_the_minus_126():
    import struct
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for code in range(16):
        f = struct.unpack("<f", struct.pack("<I", placed(code) << 16))[0]
        want = (-1.0 if code & 8 else 1.0) * e2m1[code & 7] * 2.0 ** -126
        assert f == want, (code, f, want)
