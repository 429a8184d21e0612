// Host-side launchers shared between the translation units of libqmoe (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmoe {

// route.cu
constexpr int kRouteThreads = 512;
size_t route_smem_bytes(int E);
// scratch: route_scratch_bytes(P, E) bytes of device memory (none below 8193 pairs)
size_t route_scratch_bytes(long long P, int E);
// order (optional, needs small_rows < tile_n): the tile indices with the tiles of more
// than small_rows pairs first, then the others; n_tiles[1] = the count of the first part
// The route zeroes clear_words 32-bit words from err on (the error word and any counters
// the caller places after it) before it raises a bad-id bit there: no memset is needed.
// pdl: launch its kernels with programmatic stream serialization.
int route_blocks(long long P);
cudaError_t launch_route(const int32_t* ids, int P, int E, int tile_n, int32_t* offsets,
                         int32_t* sorted_pair, int32_t* pair_pos, int32_t* tiles, int32_t* n_tiles,
                         unsigned int* err, void* scratch, cudaStream_t stream,
                         int32_t* order = nullptr, int small_rows = 0, int clear_words = 1,
                         bool pdl = false);

// misc.cu
// scale_layout: QMOE_SCALES_PLAIN, _SWIZZLED_128X4 or _PACKED_U32
cudaError_t launch_repack(const uint8_t* w, const uint8_t* s, int E, int N, int K, bool w13,
                          int scale_layout, uint8_t* out_codes, uint8_t* out_scales,
                          cudaStream_t stream);
// pdl: launch with programmatic stream serialization (see pdl_attribute)
// xs[pair_pos[i]] = x[i / top_k] for every routed pair i (pair_pos[i] >= 0)
cudaError_t launch_gather(const void* x, const int32_t* pair_pos, int M, int top_k, int H,
                          void* xs, int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_combine(const float* ypart, const int32_t* ids, int M, int top_k, int E, int H,
                           void* out, int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_selftest_dequant(uint16_t* out, cudaStream_t stream);
cudaError_t launch_selftest_timeout(unsigned int* err, long long limit_ns, cudaStream_t stream);

// gemm.cu
struct GemmParams {
  const uint8_t* wcodes;      // repacked codes
  const uint8_t* wscales;     // repacked scales
  const float* gscale;        // [E]
  const int32_t* tiles;       // [n_tiles][3]
  const int32_t* n_tiles;     // [1]
  int K;                      // contraction length
  int nrb;                    // 128-row weight blocks per expert
  // FC1 output: h [rows][I] bf16; the SwiGLU limit (+infinity: none)
  void* h;
  int I;
  float swiglu_limit;
  // FC2 output: ypart [pairs][H] fp32
  float* ypart;
  const int32_t* sorted_pair;
  const float* topk_w;
  int H;
  unsigned int* err;
  // decode schedule (stream-K): fp32 partial accumulators of units split between CTAs,
  // [CTA][2 slots][128 rows][16 pairs], and one arrival counter per (split unit, TMEM
  // lane quarter), [CTA holding the unit's first step][4], zero at launch
  float* sk_part;
  int* sk_cnt;
  uint32_t dq_mul[2];  // the dequant's multipliers 64, 4 (dequant_mul), as runtime values
  // which tiles the launch covers: 0 all, in tile order; with the split prefill
  // schedule's order (tile_order, n_tiles[1] = tiles of its first part) 1 the first
  // part (tiles of more than kSmallTileRows pairs), 2 the second
  const int32_t* tile_order;
  int tile_part;
};

// Largest grid of the decode schedule (its partial buffer has a slot pair per CTA).
constexpr int kMaxSkCtas = 192;
// Bytes of the decode schedule's partial buffer and of its counters for one GEMM.
inline size_t sk_part_bytes() { return (size_t)kMaxSkCtas * 2 * 128 * 16 * sizeof(float); }
inline size_t sk_cnt_bytes(int max_ctas) { return (size_t)max_ctas * 4 * sizeof(int); }

// Launch attribute that lets a kernel start while the previous kernel on the stream
// finishes (it must then call grid_dep_wait before reading that kernel's outputs).
// The forward uses it on every schedule but the wide prefill one, where kernels that
// take SMs early (and start their weight streams) slowed the layer by about 2%:
// measured 4.63 against 4.54 ms on the large prefill workload, while decode (0.515
// against 0.526 ms) and the narrow prefill schedule gain from the overlap.
bool forward_uses_pdl(int sched);
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

enum class GemmKind { kFc1, kFc2 };
cudaError_t launch_gemm(GemmKind kind, int sched, const CUtensorMap& tmap_b, const GemmParams& p,
                        int num_sms, cudaStream_t stream);
// Internal schedules.  kSchedPrefillNarrow: PREFILL when experts average fewer than 192
// pairs; the route cuts tiles of up to 192 pairs and orders them into two parts, and
// each GEMM runs as two launches: the tiles of more than kSmallTileRows pairs on the
// prefill kernel (two accumulators), the others on kSchedPrefillSmall, the decode
// kernel's weight-streaming pipeline with tiles of up to 64 pairs.
constexpr int kSchedPrefillNarrow = 16;
constexpr int kSchedPrefillSmall = 17;
constexpr int kSmallTileRows = 64;
int gemm_tile_n(int sched);  // max pairs per tile for a schedule
// Prefill GEMM on CTA pairs (two SMs per M = 256 tile, gemm2.cu); needs an even number
// of 128-row weight blocks (p.nrb).
cudaError_t launch_gemm2(GemmKind kind, const CUtensorMap& tmap_b, const GemmParams& p, int num_sms,
                         cudaStream_t stream);
// Rows and 64-wide slabs of the pair-row box the GEMM of a schedule loads: a 3-D box
// {64 elements, rows, slabs} per pipeline step, or (slabs 0) 2-D boxes of rows x 64
// elements.
int gemm_b_box_rows(int sched);
int gemm_b_box_slabs(int sched);

}  // namespace qmoe
