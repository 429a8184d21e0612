// GEMM epilogue for chunks of 16 accumulator columns (pairs c0 .. c0+15 of a tile) of
// one TMEM lane quarter: the lane holds weight row q*32 + lane of row block rb.
//   FC1: lanes 0..15 hold up rows, lanes 16..31 the gate rows of the same 16
//        intermediate indices; h = bf16(SiLU(gate) * up) of each valid pair.
//   FC2: ypart[pair][row] = acc * global scale * routing weight.
// gsc is the expert's global scale times 2^7 (undoing the dequant's 2^-7).
//
// epilogue_chunk_fc1 computes its 8 column results independently of each other and
// free of branches: on the prefill schedule the epilogue of a unit stalls the MMA (one
// accumulator per unit), so it must run at instruction throughput, not at the latency
// of one column at a time.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "launch.h"

namespace qmoe {

// SiLU(g) * up with e^-g taken as 2^(-g log2 e) and one approximate division; the
// result is rounded to bf16 afterwards.  For g below about -88, e^-g overflows and the
// value returned is 0 (the exact value is below 1e-36).
__device__ __forceinline__ float silu_mul(float gate, float up) {
  const float e = exp2f(gate * -1.4426950408889634f);
  return __fdividef(gate, 1.0f + e) * up;
}

// The GLM form of the SwiGLU (megamoe_rm.cu page, fc1_rm epilogue): gate clamped from
// above and up to [-limit, limit] before SiLU(gate) * up.  CLAMP false leaves both.
template <bool CLAMP>
__device__ __forceinline__ void swiglu_clamp(float& gate, float& up, float limit) {
  if constexpr (CLAMP) {
    gate = fminf(gate, limit);
    up = fminf(fmaxf(up, -limit), limit);
  }
}

template <bool CLAMP = false>
__device__ __forceinline__ void epilogue_chunk_fc1(const GemmParams& p, const float (&v)[16],
                                                   int lane, int q, int rb, int start, int rows,
                                                   int c0, float gsc) {
  // For each pair of columns (c, c+1) the lanes trade one value so that lane j < 16
  // forms h(i, c) and lane j + 16 forms h(i, c+1): every lane computes and stores.
  const bool is_up = lane < 16;
  const int i = rb * 64 + q * 16 + (lane & 15);
  // every operand read before the first store: a store through a plain pointer could
  // alias anything read through one afterwards, which would serialise each store
  // behind a reload
  __nv_bfloat16* const hp = reinterpret_cast<__nv_bfloat16*>(p.h);
  const size_t I = (size_t)p.I;
  float hv[8];
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float send = (is_up ? v[c + 1] : v[c]) * gsc;
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    float up = is_up ? v[c] * gsc : recv;
    float gate = is_up ? recv : v[c + 1] * gsc;
    swiglu_clamp<CLAMP>(gate, up, p.swiglu_limit);
    hv[c >> 1] = silu_mul(gate, up);
  }
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const int col = c0 + c + (is_up ? 0 : 1);
    if (col < rows) hp[(size_t)(start + col) * I + i] = __float2bfloat16_rn(hv[c >> 1]);
  }
}

// epilogue_chunk_fc1 through a per-warp shared tile [16 pairs][16 intermediate indices]
// bf16 (512 bytes): the h values go in as one 16-bit store each (the two half-warps
// fill rows 32 bytes apart, no bank conflicts) and come out as 16-byte rows, so each
// lane writes one 16-byte piece of a pair's h row: one global store per lane and
// chunk instead of eight 2-byte ones (global store issue dominates this epilogue).
template <bool CLAMP = false>
__device__ __forceinline__ void epilogue_chunk_fc1_tr(const GemmParams& p, const float (&v)[16],
                                                      int lane, int q, int rb, int start, int rows,
                                                      int c0, float gsc, uint8_t* tile) {
  const bool is_up = lane < 16;
  float hv[8];
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float send = (is_up ? v[c + 1] : v[c]) * gsc;
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    float up = is_up ? v[c] * gsc : recv;
    float gate = is_up ? recv : v[c + 1] * gsc;
    swiglu_clamp<CLAMP>(gate, up, p.swiglu_limit);
    hv[c >> 1] = silu_mul(gate, up);
  }
  __nv_bfloat16* const t = reinterpret_cast<__nv_bfloat16*>(tile) + (lane & 15);
#pragma unroll
  for (int m = 0; m < 8; ++m) t[(2 * m + (is_up ? 0 : 1)) * 16] = __float2bfloat16_rn(hv[m]);
  __syncwarp();
  const int col = lane >> 1, half = lane & 1;
  const uint4 w = *reinterpret_cast<const uint4*>(tile + col * 32 + half * 16);
  __nv_bfloat16* const hp = reinterpret_cast<__nv_bfloat16*>(p.h);
  if (c0 + col < rows)
    *reinterpret_cast<uint4*>(hp + (size_t)(start + c0 + col) * p.I + rb * 64 + q * 16 + half * 8) = w;
  __syncwarp();  // the tile is rewritten by the next chunk
}

// FC2 chunk with the tile's pair ids and scaled routing weights staged in shared
// memory by the same warp (st_pair / st_w, indexed by column): no global load on the
// chunk's path.
__device__ __forceinline__ void epilogue_chunk_fc2_staged(const GemmParams& p, const float (&v)[16],
                                                          int lane, int q, int rb, int rows,
                                                          int c0, const int* st_pair,
                                                          const float* st_w) {
  const int jrow = rb * 128 + q * 32 + lane;
  // every operand read before the first store (see epilogue_chunk_fc1)
  float* const yp = p.ypart;
  const size_t H = (size_t)p.H;
  int pr[16];
  float w[16];
#pragma unroll
  for (int c = 0; c < 16; c += 4) {
    *reinterpret_cast<int4*>(pr + c) = *reinterpret_cast<const int4*>(st_pair + c0 + c);
    *reinterpret_cast<float4*>(w + c) = *reinterpret_cast<const float4*>(st_w + c0 + c);
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    if (c0 + c < rows) yp[(size_t)pr[c] * H + jrow] = v[c] * w[c];
  }
}

// Stage a tile's pair ids and routing weights x gsc for epilogue_chunk_fc2_staged (one
// warp; the caller synchronises the warp before reading them back).
__device__ __forceinline__ void epilogue_stage_fc2(const GemmParams& p, int lane, int start, int rows,
                                                   float gsc, int* st_pair, float* st_w) {
  for (int j = lane; j < rows; j += 32) {
    const int pr = p.sorted_pair[start + j];
    st_pair[j] = pr;
    st_w[j] = p.topk_w[pr] * gsc;
  }
}

// Chunk epilogue that reads the chunk's pair ids and routing weights itself (FC2) and
// forms the SiLU with expf and an IEEE division (FC1).  The decode schedule uses it for
// both GEMMs (there the epilogue overlaps the next unit's MMAs, and this form kept the
// dequant loop fastest), the prefill schedules for FC2.
template <bool FC1, bool CLAMP = false>
__device__ __forceinline__ void epilogue_chunk_small(const GemmParams& p, const float (&v)[16],
                                                     int lane, int q, int rb, int start, int rows,
                                                     int c0, float gsc) {
  if constexpr (FC1) {
    // lanes 0..15 hold up rows, lanes 16..31 the gate rows of the same 16
    // intermediate indices.  For each pair of columns (c, c+1) the lanes trade
    // one value so that lane j < 16 forms h(i, c) and lane j + 16 forms
    // h(i, c+1): every lane computes and stores.
    const bool is_up = lane < 16;
    const int i = rb * 64 + q * 16 + (lane & 15);
    __nv_bfloat16* hp = reinterpret_cast<__nv_bfloat16*>(p.h);
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const float send = (is_up ? v[c + 1] : v[c]) * gsc;
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      float up = is_up ? v[c] * gsc : recv;
      float gate = is_up ? recv : v[c + 1] * gsc;
      swiglu_clamp<CLAMP>(gate, up, p.swiglu_limit);
      const int col = c0 + c + (is_up ? 0 : 1);
      if (col < rows) {
        const float hv = gate / (1.0f + expf(-gate)) * up;
        hp[(size_t)(start + col) * p.I + i] = __float2bfloat16_rn(hv);
      }
    }
  } else {
    // the chunk's 16 pair ids and routing weights: one coalesced load, then
    // broadcast by shuffles
    const int cl = lane & 15;
    int my_pair = 0;
    float my_w = 0.f;
    if (c0 + cl < rows) {
      my_pair = p.sorted_pair[start + c0 + cl];
      my_w = p.topk_w[my_pair] * gsc;
    }
    const int jrow = rb * 128 + q * 32 + lane;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int pair = __shfl_sync(0xffffffffu, my_pair, c);
      const float w = __shfl_sync(0xffffffffu, my_w, c);
      if (c0 + c < rows) p.ypart[(size_t)pair * p.H + jrow] = v[c] * w;
    }
  }
}

}  // namespace qmoe
