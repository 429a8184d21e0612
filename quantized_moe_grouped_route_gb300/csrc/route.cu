// route_sort: group the (token, expert) pairs by expert.
//
// Definition (megamoe_rm.cu page, route_prep): a pair's slot is its rank among
// earlier pairs with the same expert; pairs with expert -1 are skipped.  Offsets
// per expert follow the "total tokens including expert" prefix of cutlass
// discussion 2855.  The tile list cuts each expert's run of positions into tiles of
// at most tile_n pairs, experts ascending.
//
// Warps of 32 lanes; each owns a contiguous range of pairs, the ranges in pair order,
// so ranks come out stable without any ordering between warps:
//   A. warp-aggregated histogram: lanes with equal expert ids find each other with
//      match.any, the lowest such lane adds the group size to the warp's own row
//      of a [16][E] count table (no atomics, no races);
//   B. block scan: per-expert totals, an exclusive scan over experts (offsets), an
//      exclusive scan of tile counts, and each warp's starting position per expert;
//   C. scatter: each warp walks its range again; a pair's position is its warp's
//      running base for the expert plus its rank among equal lanes of the step.
// Up to 8192 pairs this is one block of 16 warps with the count table in shared memory
// (one launch: the decode case is launch-latency bound).  Larger inputs run A, B and C
// as three kernels: A and C over up to 152 blocks (about 256 pairs per warp), with the
// [blocks * 16][E] table in the workspace, B in one block.
#include "common.cuh"
#include "launch.h"

namespace qmoe {
namespace {

constexpr int kWarps = kRouteThreads / 32;
constexpr int kBatch = 8;  // 32-pair steps whose ids a warp loads at once

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix and
// writes the block total to *total.  `scratch` holds kWarps ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scratch[w] = incl;
  __syncthreads();
  if (w == 0) {
    int s = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += t;
    }
    if (lane < kWarps) scratch[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int excl = incl - v + (w ? scratch[w - 1] : 0);
  *total = scratch[kWarps - 1];
  __syncthreads();
  return excl;
}

// A. warp-aggregated histogram of the pairs [lo, hi) into the warp's row hw[E]:
// lanes with equal expert ids find each other with match.any and the lowest such lane
// adds the group size.  The ids of kBatch steps are loaded before the first is used,
// so a warp waits for global memory once per batch, not per step.  Returns whether an
// id >= E was seen.
__device__ __forceinline__ bool warp_histogram(const int32_t* __restrict__ ids, int lo, int hi, int E,
                                               int* hw, int lane) {
  bool bad = false;
  for (int base0 = lo; base0 < hi; base0 += 32 * kBatch) {
    int eb[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = base0 + 32 * k + lane;
      eb[k] = i < hi ? ids[i] : -1;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      int e = eb[k];
      if (e >= E) {
        bad = true;
        e = -1;
      }
      if (e < 0) e = -1;
      const unsigned m = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(m) - 1) hw[e] += __popc(m);
      __syncwarp();
    }
  }
  return bad;
}

// B. From the R per-warp rows h[R][E] of counts (rows in pair order): offsets, the tile
// list, and each row turned into that warp's first position per expert.  Thread t owns
// experts [t*ept, (t+1)*ept).  Whole block; h in shared or global memory.
// With `order` (the forward's split prefill schedule) it also lists the tile indices
// with the tiles of more than `small_rows` pairs first and the others after them, each
// part in tile order, and stores the count of the first part in n_tiles[1].
__device__ __forceinline__ void route_scan(int* h, int R, int E, int T, int32_t* __restrict__ offsets,
                                           int32_t* __restrict__ tiles, int32_t* __restrict__ n_tiles,
                                           int* scan_scratch, int32_t* __restrict__ order = nullptr,
                                           int small_rows = 0) {
  const int tid = threadIdx.x;
  const int ept = (E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = tid * ept;
  int my_pairs = 0, my_tiles = 0, my_small = 0;
  for (int j = 0; j < ept; ++j) {
    const int e = e0 + j;
    if (e < E) {
      int c = 0;
      for (int r = 0; r < R; ++r) c += h[(size_t)r * E + e];
      my_pairs += c;
      my_tiles += (c + T - 1) / T;
      // every tile of an expert holds T pairs but the last, which holds c - T (n - 1)
      if (c > 0 && c - T * ((c - 1) / T) <= small_rows) ++my_small;
    }
  }
  int total_pairs, total_tiles;
  int pair_base = block_exclusive_scan(my_pairs, scan_scratch, &total_pairs);
  int tile_base = block_exclusive_scan(my_tiles, scan_scratch, &total_tiles);
  int wide_base = 0, small_base = 0, total_small = 0;
  if (order) {
    small_base = block_exclusive_scan(my_small, scan_scratch, &total_small);
    wide_base = tile_base - small_base;  // wide tiles of the experts before this thread's
  }
  const int total_wide = total_tiles - total_small;
  for (int j = 0; j < ept; ++j) {
    const int e = e0 + j;
    if (e >= E) break;
    offsets[e] = pair_base;
    int run = pair_base;
    for (int r = 0; r < R; ++r) {
      const int c = h[(size_t)r * E + e];
      h[(size_t)r * E + e] = run;  // becomes warp r's next position for expert e
      run += c;
    }
    const int cnt = run - pair_base;
    for (int s = 0; s < cnt; s += T) {
      const int rows = min(T, cnt - s);
      tiles[3 * tile_base + 0] = e;
      tiles[3 * tile_base + 1] = pair_base + s;
      tiles[3 * tile_base + 2] = rows;
      if (order) {
        if (rows <= small_rows)
          order[total_wide + small_base++] = tile_base;
        else
          order[wide_base++] = tile_base;
      }
      ++tile_base;
    }
    pair_base = run;
  }
  if (tid == 0) {
    offsets[E] = total_pairs;
    n_tiles[0] = total_tiles;
    if (order) n_tiles[1] = total_wide;
  }
}

// C. stable scatter of the pairs [lo, hi) from the warp's running positions hw[E]
// (steps in order within each batch, batches in order).
__device__ __forceinline__ void warp_scatter(const int32_t* __restrict__ ids, int lo, int hi, int E,
                                             int* hw, int lane, int32_t* __restrict__ sorted_pair,
                                             int32_t* __restrict__ pair_pos) {
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base0 = lo; base0 < hi; base0 += 32 * kBatch) {
    int eb[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = base0 + 32 * k + lane;
      eb[k] = i < hi ? ids[i] : -1;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = base0 + 32 * k + lane;
      int e = eb[k];
      if (e >= E || e < 0) e = -1;
      const unsigned m = __match_any_sync(0xffffffffu, e);
      const int b = e >= 0 ? hw[e] : 0;
      const int pos = b + __popc(m & lt_mask);
      __syncwarp();
      if (e >= 0 && lane == __ffs(m) - 1) hw[e] = b + __popc(m);
      __syncwarp();
      if (i < hi) {
        if (e >= 0) {
          sorted_pair[pos] = i;
          pair_pos[i] = pos;
        } else {
          pair_pos[i] = -1;
        }
      }
    }
  }
}

// Pairs per warp: contiguous ranges of whole 32-pair steps, in pair order over the
// warps of all blocks (warp g = block * kWarps + warp), so ranks come out stable.
__host__ __device__ __forceinline__ int route_chunk(int P, int nwarps) {
  return (((P + nwarps - 1) / nwarps) + 31) & ~31;
}

// Small inputs: the whole route in one block of kWarps warps, rows in shared memory.
// clear_words 32-bit words from err on are zeroed first (the error word and, in a
// forward, the GEMMs' split-unit counters), so that no memset has to run before the
// route.  Launched with programmatic serialization, the block waits for the
// stream's previous kernel before touching any output, and lets the next kernel (the
// gather) start its set-up at once.
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const int32_t* __restrict__ ids, int P, int E, int T, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ sorted_pair, int32_t* __restrict__ pair_pos,
                 int32_t* __restrict__ tiles, int32_t* __restrict__ n_tiles,
                 unsigned int* __restrict__ err, int32_t* __restrict__ order, int small_rows,
                 int clear_words) {
  extern __shared__ int hist[];  // [kWarps][E]
  __shared__ int scan_scratch[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  grid_dep_wait();
  grid_dep_launch();
  for (int i = tid; i < clear_words; i += kRouteThreads) err[i] = 0u;
  for (int i = tid; i < kWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();
  const int chunk = route_chunk(P, kWarps);
  const int lo = w * chunk;
  const int hi = min(P, lo + chunk);
  int* hw = hist + w * E;
  if (warp_histogram(ids, lo, hi, E, hw, lane)) atomicOr(err, QMOE_FLAG_BAD_ID);
  __syncthreads();
  route_scan(hist, kWarps, E, T, offsets, tiles, n_tiles, scan_scratch, order, small_rows);
  __syncthreads();
  warp_scatter(ids, lo, hi, E, hw, lane, sorted_pair, pair_pos);
  for (int pos = offsets[E] + tid; pos < P; pos += kRouteThreads) sorted_pair[pos] = -1;
}

// Large inputs, three kernels over `blocks` blocks of kWarps warps; the per-warp rows
// live in global memory (gh [blocks * kWarps][E]), each block's bad-id flag in gbad
// [blocks] after them.  The scan kernel (one block) zeroes the clear_words words from
// err on and then raises the bad-id bit from the blocks' flags, so that no memset has to
// run before the route.  Launched with programmatic serialization, each kernel waits
// for its predecessor before touching any output and lets its successor be scheduled.
__global__ void __launch_bounds__(kRouteThreads)
    route_hist_kernel(const int32_t* __restrict__ ids, int P, int E, int* __restrict__ gh,
                      int* __restrict__ gbad) {
  extern __shared__ int hist[];  // [kWarps][E]
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  grid_dep_wait();
  grid_dep_launch();
  if (tid == 0) bad = 0;
  for (int i = tid; i < kWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();
  const int chunk = route_chunk(P, gridDim.x * kWarps);
  const int lo = min(P, (blockIdx.x * kWarps + w) * chunk);
  const int hi = min(P, lo + chunk);
  if (warp_histogram(ids, lo, hi, E, hist + w * E, lane)) bad = 1;
  __syncthreads();
  int* dst = gh + (size_t)blockIdx.x * kWarps * E;
  for (int i = tid; i < kWarps * E; i += kRouteThreads) dst[i] = hist[i];
  if (tid == 0) gbad[blockIdx.x] = bad;
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    route_scan_kernel(int R, int E, int T, int* __restrict__ gh, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ tiles, int32_t* __restrict__ n_tiles,
                      int32_t* __restrict__ order, int small_rows, const int* __restrict__ gbad,
                      int nblocks, unsigned int* __restrict__ err, int clear_words) {
  __shared__ int scan_scratch[kWarps];
  const int tid = threadIdx.x;
  grid_dep_wait();
  grid_dep_launch();
  for (int i = tid; i < clear_words; i += kRouteThreads) err[i] = 0u;
  int any = 0;
  for (int b = tid; b < nblocks; b += kRouteThreads) any |= gbad[b];
  if (__syncthreads_or(any) && tid == 0) atomicOr(err, QMOE_FLAG_BAD_ID);
  route_scan(gh, R, E, T, offsets, tiles, n_tiles, scan_scratch, order, small_rows);
}

__global__ void __launch_bounds__(kRouteThreads)
    route_scatter_kernel(const int32_t* __restrict__ ids, int P, int E, const int* __restrict__ gh,
                         const int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair,
                         int32_t* __restrict__ pair_pos) {
  extern __shared__ int hist[];  // [kWarps][E]: this block's warps' first positions
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  grid_dep_wait();
  grid_dep_launch();
  const int* src = gh + (size_t)blockIdx.x * kWarps * E;
  for (int i = tid; i < kWarps * E; i += kRouteThreads) hist[i] = src[i];
  __syncthreads();
  const int chunk = route_chunk(P, gridDim.x * kWarps);
  const int lo = min(P, (blockIdx.x * kWarps + w) * chunk);
  const int hi = min(P, lo + chunk);
  warp_scatter(ids, lo, hi, E, hist + w * E, lane, sorted_pair, pair_pos);
  for (int pos = offsets[E] + blockIdx.x * kRouteThreads + tid; pos < P;
       pos += gridDim.x * kRouteThreads)
    sorted_pair[pos] = -1;
}

}  // namespace

size_t route_smem_bytes(int E) { return (size_t)kWarps * (size_t)E * sizeof(int); }

// Blocks of the multi-block route: about 256 pairs per warp (one batch of steps), at
// most 152 blocks; inputs of up to 8192 pairs take the one-block kernel.
int route_blocks(long long P) {
  if (P <= 8192) return 1;
  const long long b = (P + (long long)kWarps * 256 - 1) / ((long long)kWarps * 256);
  return (int)(b < 152 ? b : 152);
}

size_t route_scratch_bytes(long long P, int E) {
  const int b = route_blocks(P);
  return b > 1 ? (size_t)b * (kWarps * (size_t)E + 1) * sizeof(int) : 0;
}

cudaError_t launch_route(const int32_t* ids, int P, int E, int tile_n, int32_t* offsets,
                         int32_t* sorted_pair, int32_t* pair_pos, int32_t* tiles, int32_t* n_tiles,
                         unsigned int* err, void* scratch, cudaStream_t stream, int32_t* order,
                         int small_rows, int clear_words, bool pdl) {
  const size_t smem = route_smem_bytes(E);
  const int blocks = route_blocks(P);
  if (blocks == 1) {
    cudaError_t rc = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
    if (rc != cudaSuccess) return rc;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, route_kernel, ids, P, E, tile_n, offsets, sorted_pair,
                              pair_pos, tiles, n_tiles, err, order, small_rows, clear_words);
  }
  int* gh = reinterpret_cast<int*>(scratch);
  int* gbad = gh + (size_t)blocks * kWarps * E;
  cudaError_t rc = cudaFuncSetAttribute(route_hist_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (rc == cudaSuccess)
    rc = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
  if (rc != cudaSuccess) return rc;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.blockDim = dim3(kRouteThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.gridDim = dim3(blocks);
  cfg.dynamicSmemBytes = smem;
  rc = cudaLaunchKernelEx(&cfg, route_hist_kernel, ids, P, E, gh, gbad);
  if (rc != cudaSuccess) return rc;
  cfg.gridDim = dim3(1);
  cfg.dynamicSmemBytes = 0;
  rc = cudaLaunchKernelEx(&cfg, route_scan_kernel, blocks * kWarps, E, tile_n, gh, offsets, tiles,
                          n_tiles, order, small_rows, (const int*)gbad, blocks, err, clear_words);
  if (rc != cudaSuccess) return rc;
  cfg.gridDim = dim3(blocks);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, route_scatter_kernel, ids, P, E, (const int*)gh,
                            (const int32_t*)offsets, sorted_pair, pair_pos);
}

}  // namespace qmoe
