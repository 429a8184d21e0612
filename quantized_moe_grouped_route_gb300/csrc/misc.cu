// Repack, activation gather, top_k combine and the diagnostic kernels.
#include "common.cuh"
#include "dequant.cuh"
#include "launch.h"

namespace qmoe {
namespace {

// Repacked layout, per (expert e, 128-row block rb, 128-wide K step ks):
//   codes : 8192 bytes = [kk 0..3][row 0..127][16 bytes = 32 elements], each 4-byte
//           word holding eight consecutive K elements in the pack_codes8 layout
//   scales: 1024 bytes = [row 0..127][8 scale bytes of the step's 8 K blocks]
// so one stage of the GEMM is two contiguous bulk copies, and each dequant thread
// (one weight row) reads its 16-byte chunks and its 8 scale bytes without shared
// memory bank conflicts.
__global__ void repack_codes_kernel(const uint8_t* __restrict__ w, int E, int N, int K, int w13,
                                    uint32_t* __restrict__ out) {
  const int nrb = N / 128, nks = K / 128;
  const long long total = (long long)E * N * (K / 8);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int wd = (int)(idx & 3);
    const int r = (int)((idx >> 2) & 127);
    long long rest = idx >> 9;
    const int kk = (int)(rest & 3);
    rest >>= 2;
    const int ks = (int)(rest % nks);
    rest /= nks;
    const int rb = (int)(rest % nrb);
    const int e = (int)(rest / nrb);
    const int n = repack_row(w13 != 0, N, rb, r);
    const int k0 = ks * 128 + kk * 32 + wd * 8;
    const uint32_t plain =
        *reinterpret_cast<const uint32_t*>(w + ((size_t)e * N + n) * (size_t)(K / 2) + k0 / 2);
    out[idx] = pack_codes8(plain);
  }
}

// layout of the input scales (QMOE_SCALES_*):
//  PLAIN          [E][N][K/16] bytes;
//  SWIZZLED_128X4 the 128x4 swizzle of CUTLASS / FlashInfer NVFP4 weights (megamoe_rm.cu
//                 page, scale_off): per expert, tiles of 128 rows x 4 scales, 512 bytes
//                 each, the 4-column tile index fastest; inside a tile, row r's 4
//                 scales at (r % 32) * 16 + ((r / 32) % 4) * 4.  A row's 8 scales of one
//                 128-wide K block are then two 4-byte words, 512 bytes apart;
//  PACKED_U32     [E][N][K/64] uint32 words (tilelang_kernels.py page,
//                 grouped_gemm_fp4_packed_sf), scale j of word g (K block 4g + j) in
//                 bits 8j..8j+7: a 128-wide K block's 8 scales are words 2ks, 2ks + 1.
__global__ void repack_scales_kernel(const uint8_t* __restrict__ s, int E, int N, int K, int w13,
                                     int layout, uint2* __restrict__ out) {
  const int nrb = N / 128, nks = K / 128;
  const long long total = (long long)E * N * nks;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx & 127);
    long long rest = idx >> 7;
    const int ks = (int)(rest % nks);
    rest /= nks;
    const int rb = (int)(rest % nrb);
    const int e = (int)(rest / nrb);
    const int n = repack_row(w13 != 0, N, rb, r);
    const size_t C = (size_t)(K / 16);
    if (layout == QMOE_SCALES_PACKED_U32) {
      const uint32_t* wrow = reinterpret_cast<const uint32_t*>(s) + ((size_t)e * N + n) * (C / 4);
      // output byte b of the step = scale of K block 8 ks + b (bits 8b.. of the words)
      uint32_t o[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t wv = wrow[2 * ks + h];
        o[h] = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[h] |= ((wv >> (8 * j)) & 0xFFu) << (8 * j);
      }
      out[idx] = make_uint2(o[0], o[1]);
    } else if (layout == QMOE_SCALES_SWIZZLED_128X4) {
      const uint8_t* se = s + (size_t)e * N * C;
      const size_t o = ((size_t)(n >> 7) * (C >> 2) + (size_t)ks * 2) * 512 + (size_t)(n & 31) * 16 +
                       (size_t)((n >> 5) & 3) * 4;
      uint2 v;
      v.x = *reinterpret_cast<const uint32_t*>(se + o);
      v.y = *reinterpret_cast<const uint32_t*>(se + o + 512);
      out[idx] = v;
    } else {
      out[idx] = *reinterpret_cast<const uint2*>(s + ((size_t)e * N + n) * C + ks * 8);
    }
  }
}

// xs[pair_pos[m * top_k + k]] = x[m] for every routed pair, 16-byte chunks.  Work items
// are (token, segment of 256 chunks) taken one per warp: the warp reads its segment of
// the token's row once (eight 16-byte chunks per lane) and writes it to the position of
// each of the token's routed pairs, so x is read in one pass however many of its slots
// a token routes (reading it per pair in expert order re-read each row top_k times,
// mostly from L2 but not always).
__global__ void gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ pair_pos,
                              int M, int top_k, int chunks, uint4* __restrict__ xs) {
  grid_dep_wait();    // the route's outputs
  grid_dep_launch();  // FC1 may start streaming weights
  constexpr int kSeg = 256, kPer = kSeg / 32;
  const int nseg = (chunks + kSeg - 1) / kSeg;
  const long long items = (long long)M * nseg;
  const int lane = threadIdx.x & 31;
  const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long it = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items;
       it += warps) {
    const int m = (int)(it / nseg);
    const int c0 = (int)(it - (long long)m * nseg) * kSeg;
    const uint4* src = x + (size_t)m * chunks;
    uint4 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int c = c0 + lane + 32 * j;
      if (c < chunks) v[j] = src[c];
    }
    for (int k = 0; k < top_k; ++k) {
      const int pos = pair_pos[(size_t)m * top_k + k];
      if (pos < 0) continue;
      uint4* dst = xs + (size_t)pos * chunks;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int c = c0 + lane + 32 * j;
        if (c < chunks) dst[c] = v[j];
      }
    }
  }
}

// out[m][j] = bf16( sum over k ascending of ypart[m*top_k + k][j] ) over the slots
// whose expert id is in [0, E) (megamoe_rm.cu page, combine).  Fixed order, no
// atomics: deterministic.  8 columns per thread.
__global__ void combine_kernel(const float* __restrict__ ypart, const int32_t* __restrict__ ids,
                               int M, int top_k, int E, int H, uint4* __restrict__ out) {
  grid_dep_wait();    // FC2's partial rows
  grid_dep_launch();  // the stream's next kernel (the next layer's route) may be scheduled
  const int c8 = H / 8;
  const long long total = (long long)M * c8;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(idx / c8);
    const int j0 = (int)(idx - (long long)m * c8) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < top_k; ++k) {
      const int e = ids[m * top_k + k];
      if (e < 0 || e >= E) continue;
      const float4* src = reinterpret_cast<const float4*>(ypart + ((size_t)m * top_k + k) * H + j0);
      const float4 a = src[0], b = src[1];
      acc[0] += a.x;
      acc[1] += a.y;
      acc[2] += a.z;
      acc[3] += a.w;
      acc[4] += b.x;
      acc[5] += b.y;
      acc[6] += b.z;
      acc[7] += b.w;
    }
    uint4 o;
    __nv_bfloat162 t0 = __floats2bfloat162_rn(acc[0], acc[1]);
    __nv_bfloat162 t1 = __floats2bfloat162_rn(acc[2], acc[3]);
    __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[4], acc[5]);
    __nv_bfloat162 t3 = __floats2bfloat162_rn(acc[6], acc[7]);
    o.x = *reinterpret_cast<uint32_t*>(&t0);
    o.y = *reinterpret_cast<uint32_t*>(&t1);
    o.z = *reinterpret_cast<uint32_t*>(&t2);
    o.w = *reinterpret_cast<uint32_t*>(&t3);
    out[idx] = o;
  }
}

// Every (code, scale) pair at every element position of a packed word, through the
// GEMM's dequant path (with its multipliers passed in at run time, as the GEMM gets
// them).  Thread c fills the word with codes (c + j) mod 16 at positions j = 0..7, so
// each position meets all 16 codes beside 7 other nonzero codes.
__global__ void selftest_dequant_kernel(uint16_t* __restrict__ out, DequantMul dqm) {
  const int sb = blockIdx.x;  // scale byte
  const int c = threadIdx.x;  // 0..15
  if (c >= 16) return;
  const uint32_t s2 = e4m3_scale_bf16x2(sb);
  uint32_t plain = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) plain |= (uint32_t)((c + j) & 15) << (4 * j);
  uint32_t o[4];
  dequant8(pack_codes8(plain), s2, o, dqm);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint16_t v = (j & 1) ? (uint16_t)(o[j >> 1] >> 16) : (uint16_t)(o[j >> 1] & 0xFFFF);
    // undo the 2^-7 the kernels fold into the epilogue: multiply by 128 exactly
    const float f = __bfloat162float(__ushort_as_bfloat16(v)) * 128.0f;
    out[((size_t)c * 256 + sb) * 8 + j] = __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
}

// One bounded wait on a barrier that nothing ever arrives at.
__global__ void selftest_timeout_kernel(unsigned int* err, long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
  }
  __syncthreads();
}

int grid_for(long long work, int threads, int num_sms) {
  long long b = (work + threads - 1) / threads;
  long long cap = (long long)num_sms * 8;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

cudaError_t launch_repack(const uint8_t* w, const uint8_t* s, int E, int N, int K, bool w13,
                          int scale_layout, uint8_t* out_codes, uint8_t* out_scales,
                          cudaStream_t stream) {
  const long long words = (long long)E * N * (K / 8);
  const long long rows = (long long)E * N * (K / 128);
  repack_codes_kernel<<<grid_for(words, 256, 1184), 256, 0, stream>>>(
      w, E, N, K, w13 ? 1 : 0, reinterpret_cast<uint32_t*>(out_codes));
  cudaError_t rc = cudaGetLastError();
  if (rc != cudaSuccess) return rc;
  repack_scales_kernel<<<grid_for(rows, 256, 1184), 256, 0, stream>>>(
      s, E, N, K, w13 ? 1 : 0, scale_layout, reinterpret_cast<uint2*>(out_scales));
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x, const int32_t* pair_pos, int M, int top_k, int H,
                          void* xs, int num_sms, cudaStream_t stream, bool pdl) {
  const int chunks = H / 8;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  // a warp per (token, 256-chunk segment)
  cfg.gridDim = dim3(grid_for((long long)M * ((chunks + 255) / 256) * 32, 256, num_sms));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_kernel, reinterpret_cast<const uint4*>(x), pair_pos, M,
                            top_k, chunks, reinterpret_cast<uint4*>(xs));
}

cudaError_t launch_combine(const float* ypart, const int32_t* ids, int M, int top_k, int E, int H,
                           void* out, int num_sms, cudaStream_t stream, bool pdl) {
  const long long work = (long long)M * (H / 8);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(grid_for(work, 256, num_sms));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, ypart, ids, M, top_k, E, H,
                            reinterpret_cast<uint4*>(out));
}

cudaError_t launch_selftest_dequant(uint16_t* out, cudaStream_t stream) {
  selftest_dequant_kernel<<<256, 32, 0, stream>>>(out, dequant_mul());
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned int* err, long long limit_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace qmoe
