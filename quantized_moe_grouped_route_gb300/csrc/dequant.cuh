// NVFP4 -> bf16 dequantization used by the grouped GEMM, and the weight layout the
// one-time repack writes for it.
//
// The value of a weight is E2M1 code * E4M3 block scale (megamoe_rm.cu page,
// chunk_mma: "hmul2(e2m1x2(..), scale)"); the product has at most 6 significant bits
// and lies in [2^-10, 2688], so it is exact in bf16.
//
// Bit placement instead of conversion: a 4-bit code s|e1 e0|m written into a bf16
// as (s << 15) | (e1 e0 m << 6) reads as code * 2^-126 (code 0.5 lands on the
// bf16 subnormal 2^-127, code 0 on zero).  Multiplying that by the bf16 constant
// scale * 2^119 gives code * scale * 2^-7 exactly; the GEMM epilogue multiplies the
// fp32 accumulator by 2^7 together with the global scale.
//
// The repack stores eight codes of one 32-bit word so that four output bf16x2 words
// come out of shifts, one rotation and masks with the mask M = 0x81C081C0 (magnitudes
// at bits 6-8 / 22-24, signs at 15 / 31):
//   elements 0,1 : magnitude at bits  6- 8 / 22-24, sign 15 / 31   -> q & M
//   elements 2,3 : magnitude at bits  0- 2 / 16-18, sign  9 / 25   -> (q << 6) & M
//   elements 4,5 : magnitude at bits 26-28 / 10-12, sign  3 / 19   -> rotl(q, 12) & M
//   elements 6,7 : magnitude bits 0,1 at 4,5 / 20,21, bit 2 at 14 / 30, sign 13 / 29
//                  -> ((q << 2) & 0x80C080C0) | ((q >> 6) & 0x01000100)
// Every bit of the word holds one bit of one code.  No packing gives each of the four
// outputs one shift (or rotation) and one mask: the target bits {6, 7, 8, 15} of a half
// tile no 32-bit word, so one output takes two pieces.  This one costs 13 instructions
// per 8 codes (7 logic, 2 multiply-adds, 4 bf16x2 multiplies), against 15 for a
// packing built from plain shifts alone.
#pragma once

#include <stdint.h>

namespace qmoe {

// Pack eight plain codes (code j in bits 4j..4j+3 of `plain`) into the layout above.
__host__ __device__ __forceinline__ uint32_t pack_codes8(uint32_t plain) {
  uint32_t q = 0;
  auto code = [&](int j) { return (plain >> (4 * j)) & 0xFu; };
  auto mag = [&](int j) { return code(j) & 7u; };
  auto sgn = [&](int j) { return (code(j) >> 3) & 1u; };
  q |= mag(0) << 6;
  q |= sgn(0) << 15;
  q |= mag(1) << 22;
  q |= sgn(1) << 31;
  q |= mag(2) << 0;
  q |= sgn(2) << 9;
  q |= mag(3) << 16;
  q |= sgn(3) << 25;
  q |= mag(4) << 26;
  q |= sgn(4) << 3;
  q |= mag(5) << 10;
  q |= sgn(5) << 19;
  q |= (mag(6) & 3u) << 4;
  q |= ((mag(6) >> 2) & 1u) << 14;
  q |= sgn(6) << 13;
  q |= (mag(7) & 3u) << 20;
  q |= ((mag(7) >> 2) & 1u) << 30;
  q |= sgn(7) << 29;
  return q;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Dequantize one packed word (eight consecutive K elements) with the broadcast
// bf16x2 constant scale * 2^119; writes four bf16x2 words in K order.
// The two left shifts q * 2^k run as integer multiply-adds, on the multiply-add pipe,
// beside the logic ops on the integer pipe.  The multipliers (64, 4) are runtime
// values (DequantMul), so that the compiler keeps them multiplies instead of turning
// them back into shifts.
struct DequantMul {
  uint32_t m64, m4;
};
__host__ __device__ constexpr DequantMul dequant_mul() { return DequantMul{64u, 4u}; }

__device__ __forceinline__ uint32_t shl_fma(uint32_t q, uint32_t pow2) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, 0;" : "=r"(r) : "r"(q), "r"(pow2));
  return r;
}

__device__ __forceinline__ void dequant8(uint32_t q, uint32_t s2, uint32_t* o, const DequantMul& m) {
  const uint32_t M = 0x81C081C0u;
  const uint32_t a0 = q & M;
  const uint32_t a1 = shl_fma(q, m.m64) & M;
  const uint32_t a2 = __funnelshift_l(q, q, 12) & M;  // rotate left by 12
  const uint32_t a3 = (shl_fma(q, m.m4) & 0x80C080C0u) | ((q >> 6) & 0x01000100u);
  o[0] = bf16x2_mul(a0, s2);
  o[1] = bf16x2_mul(a1, s2);
  o[2] = bf16x2_mul(a2, s2);
  o[3] = bf16x2_mul(a3, s2);
}

// bf16x2 broadcast of (E4M3 value of byte b) * 2^119, from the E4M3 bit fields
// (sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0, exponent 0
// subnormal, 0x7F / 0xFF NaN).  Exact: at most 4 significant bits, <= 1.75 * 2^127.
__device__ __forceinline__ uint32_t e4m3_scale_bf16x2(int b) {
  const int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  float v;
  if (e == 15 && m == 7)
    v = __int_as_float(0x7fc00000);
  else if (e == 0)
    v = ldexpf((float)m, 110);
  else
    v = ldexpf(1.0f + (float)m * 0.125f, e - 7 + 119);
  if (s) v = -v;
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return h | (h << 16);
}

// Row of the repacked 128-row block `rb` -> row of the plain weight matrix.
// w13 ([2I] rows): within each 32-row quarter q, rows 0..15 are up rows and rows
// 16..31 the gate rows of the same 16 intermediate indices, so one warp's TMEM
// lanes hold matching up/gate pairs 16 lanes apart.  w2: identity.
__host__ __device__ __forceinline__ int repack_row(bool w13, int N, int rb, int r) {
  if (!w13) return rb * 128 + r;
  const int I = N / 2;
  const int q = r >> 5, j = r & 31;
  const int i = rb * 64 + q * 16 + (j & 15);
  return j < 16 ? i : I + i;
}

}  // namespace qmoe
