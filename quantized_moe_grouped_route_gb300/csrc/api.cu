// C-ABI boundary of libqmoe: argument checks, workspace layout, tensor maps and
// the launch sequence of the layer (megamoe_rm.cu page, megamoe_rm_forward: shape
// checks, scratch carved from caller memory, everything on the caller's stream).
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "dequant.cuh"
#include "launch.h"

namespace qmoe {
namespace {

constexpr int kMaxDevices = 64;
// Per-device facts looked up once (0 = not yet known); atomics, since several host
// threads may make their first calls at the same time.
std::atomic<int> g_num_sms[kMaxDevices];
std::atomic<int> g_arch_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 unsupported

int device_info(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMOE_ERR_CUDA;
  int ok = g_arch_ok[dev].load(std::memory_order_acquire);
  if (ok == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return QMOE_ERR_CUDA;
    g_num_sms[dev].store(sms, std::memory_order_relaxed);
    ok = (major == 10 && minor == 3) ? 1 : -1;
    g_arch_ok[dev].store(ok, std::memory_order_release);
  }
  if (ok < 0) return QMOE_ERR_ARCH;
  *num_sms = g_num_sms[dev].load(std::memory_order_relaxed);
  return QMOE_OK;
}

// Driver entry points, resolved once (a function-local static is initialised once even
// when several threads get here first).
template <class Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(ptr);
  return nullptr;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn =
      driver_fn<PFN_cuTensorMapEncodeTiled_v12000>("cuTensorMapEncodeTiled");
  return fn;
}

PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
  static const PFN_cuCtxGetCurrent_v4000 fn = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent");
  return fn;
}

// Tensor map over a row-major bf16 matrix [rows][cols] for the GEMM's pair rows.
// box_slabs == 0: 2-D, box box_rows rows x 64 elements.  box_slabs > 0: 3-D view
// {64 elements, rows, cols / 64 slabs} (slab stride 128 bytes), box
// {64, box_rows, box_slabs}, which lands in shared memory as [slab][row][64 elements].
int make_tmap_rows(CUtensorMap* map, const void* base, int rows, int cols, int box_rows,
                   int box_slabs) {
  auto fn = encode_fn();
  if (!fn) return QMOE_ERR_CUDA;
  CUresult r;
  if (box_slabs == 0) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)cols / 64};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_slabs};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? QMOE_OK : QMOE_ERR_CUDA;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct ForwardLayout {
  size_t offsets, sorted_pair, pair_pos, tiles, n_tiles, route_scratch, xs, h, ypart, total;
  size_t tile_order;  // split prefill schedule: the route's two-part tile order
  // decode schedule: arrival counters of FC1 and FC2 (cleared with the error word,
  // [0, clear_bytes), by the route) and the partial accumulators of split units
  size_t sk_cnt1, sk_cnt2, clear_bytes, sk_part;
  int rows;  // rows of xs / h (>= 16, multiple of 16)
  int tile_n, max_tiles;
};

int check_shape(int M, int H, int I, int E, int top_k) {
  if (M < 0 || E < 1 || E > 2048 || top_k < 1 || top_k > 64) return QMOE_ERR_SHAPE;
  if (H < 128 || I < 128 || H % 128 || I % 128 || H > 65536 || I > 65536) return QMOE_ERR_SHAPE;
  if ((long long)M * top_k >= (1LL << 31) / 16) return QMOE_ERR_SHAPE;
  return QMOE_OK;
}

// The schedule a call runs.  PREFILL takes one of two tile shapes by the mean count
// of pairs per expert: from 192 on, tiles of up to 320 pairs with one accumulator (an
// expert's rows in one tile, the weights dequantized once per row block, the widest
// MMAs); below, tiles of up to 192 pairs, those of more than 64 pairs on the prefill
// kernel with two accumulators (the epilogue of a tile overlaps the MMAs of the next)
// and the others on the decode kernel's weight-streaming pipeline.
int resolve_sched(int sched, int M, int top_k, int E) {
  const long long P = (long long)M * top_k;
  if (sched == QMOE_SCHED_DECODE || sched == QMOE_SCHED_PREFILL_PAIR) return sched;
  if (sched == QMOE_SCHED_AUTO && P <= 4LL * E) return QMOE_SCHED_DECODE;
  return P >= 192LL * E ? QMOE_SCHED_PREFILL : kSchedPrefillNarrow;
}

ForwardLayout forward_layout(int M, int H, int I, int E, int top_k, int sched) {
  ForwardLayout L;
  const long long P = (long long)M * top_k;
  L.tile_n = gemm_tile_n(resolve_sched(sched, M, top_k, E));
  L.max_tiles = (int)((P + L.tile_n - 1) / L.tile_n) + E;
  L.rows = (int)align_up((size_t)(P > 0 ? P : 1), 16);
  const bool sk = resolve_sched(sched, M, top_k, E) == QMOE_SCHED_DECODE;
  size_t off = kWsHeaderBytes;
  L.sk_cnt1 = off;
  off += sk ? sk_cnt_bytes(kMaxSkCtas) : 0;
  L.sk_cnt2 = off;
  off += sk ? sk_cnt_bytes(kMaxSkCtas) : 0;
  L.clear_bytes = off;
  off = align_up(off, 256);
  L.sk_part = off;
  off = align_up(off + (sk ? sk_part_bytes() : 0), 256);
  L.offsets = off;
  off = align_up(off + 4 * (size_t)(E + 1), 256);
  L.sorted_pair = off;
  off = align_up(off + 4 * (size_t)P, 256);
  L.pair_pos = off;
  off = align_up(off + 4 * (size_t)P, 256);
  L.tiles = off;
  off = align_up(off + 12 * (size_t)L.max_tiles, 256);
  L.n_tiles = off;  // [2]: all tiles, tiles of the split order's first part
  off = align_up(off + 8, 256);
  L.tile_order = off;
  if (resolve_sched(sched, M, top_k, E) == kSchedPrefillNarrow)
    off = align_up(off + 4 * (size_t)L.max_tiles, 256);
  L.route_scratch = off;
  off = align_up(off + route_scratch_bytes(P, E), 1024);
  L.xs = off;
  off = align_up(off + 2 * (size_t)L.rows * H, 1024);
  L.h = off;
  off = align_up(off + 2 * (size_t)L.rows * I, 1024);
  L.ypart = off;
  off = align_up(off + 4 * (size_t)P * H, 256);
  L.total = off;
  return L;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA; }

// Scratch for moe_nvfp4_forward_noalloc: a fixed array inside the library, so that
// callers which cannot allocate device memory still have somewhere to put the
// routing tables, gathered activations, h and per-pair partial outputs.  Every GPU
// that loads the library holds it until the process exits.
__device__ __align__(256) uint8_t g_noalloc_scratch[QMOE_NOALLOC_SCRATCH_BYTES];

// Its device address.  Host code cannot use the symbol itself as a device pointer: the
// address is looked up with cudaGetSymbolAddress, which gives the address in the CUDA
// context current at the time.  It is cached per device together with that context and
// looked up again whenever the calling thread's current context differs (after
// cudaDeviceReset, or for a caller running its own context), under a lock.
struct NoallocAddr {
  CUcontext ctx;
  void* addr;
};
NoallocAddr g_noalloc_addr[kMaxDevices];
std::mutex g_noalloc_mutex;

int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMOE_ERR_CUDA;
  auto get_ctx = ctx_current_fn();
  if (!get_ctx) return QMOE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return QMOE_ERR_CUDA;  // null: no context current yet
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocAddr& c = g_noalloc_addr[dev];
  if (!ctx || c.ctx != ctx || !c.addr) {
    // the lookup makes the device's primary context current if the thread had none
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr)
      return QMOE_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return QMOE_ERR_CUDA;
    c.ctx = ctx;
    c.addr = addr;
  }
  *out = c.addr;
  return QMOE_OK;
}

}  // namespace
}  // namespace qmoe

using namespace qmoe;

extern "C" {

int qmoe_sched_tile_n(int sched, int M, int top_k, int E) {
  return gemm_tile_n(resolve_sched(sched, M, top_k, E));
}

int qmoe_forward_kernel_count(int M, int top_k, int E, int sched) {
  if (M < 0 || top_k < 1 || E < 1) return QMOE_ERR_ARG;
  if (sched < QMOE_SCHED_AUTO || sched > QMOE_SCHED_PREFILL_PAIR) return QMOE_ERR_ARG;
  if (M == 0) return 0;
  const long long P = (long long)M * top_k;
  // the route (one kernel, or three above 8192 pairs), gather, FC1, FC2, combine; the
  // split prefill schedule runs FC1 and FC2 as two launches each
  const int split = resolve_sched(sched, M, top_k, E) == kSchedPrefillNarrow ? 2 : 0;
  return 4 + split + (route_scratch_bytes(P, E) > 0 ? 3 : 1);
}

int qmoe_max_tiles(int M, int top_k, int E, int tile_n) {
  if (M < 0 || top_k < 1 || E < 1 || tile_n < 1) return QMOE_ERR_ARG;
  const long long P = (long long)M * top_k;
  return (int)((P + tile_n - 1) / tile_n) + E;
}

size_t qmoe_route_workspace_size(int M, int top_k, int E, int tile_n) {
  (void)tile_n;
  if (M < 0 || top_k < 1 || E < 1) return kWsHeaderBytes;
  return kWsHeaderBytes + route_scratch_bytes((long long)M * top_k, E);
}

int moe_route(const int32_t* topk_ids_dev, int M, int top_k, int E, int tile_n,
              int32_t* offsets_dev, int32_t* sorted_pair_dev, int32_t* pair_pos_dev,
              int32_t* tiles_dev, int32_t* n_tiles_dev, void* workspace_dev, size_t ws_bytes,
              void* stream) {
  if (M < 0 || top_k < 1 || top_k > 64 || E < 1 || E > 2048 || tile_n < 1 || tile_n > 4096)
    return QMOE_ERR_SHAPE;
  if ((long long)M * top_k >= (1LL << 31) / 16) return QMOE_ERR_SHAPE;
  if (!offsets_dev || !n_tiles_dev || !workspace_dev || !tiles_dev) return QMOE_ERR_ARG;
  if (M > 0 && (!topk_ids_dev || !sorted_pair_dev || !pair_pos_dev)) return QMOE_ERR_ARG;
  if ((uintptr_t)workspace_dev & 255) return QMOE_ERR_ARG;
  if (ws_bytes < qmoe_route_workspace_size(M, top_k, E, tile_n)) return QMOE_ERR_WORKSPACE;
  int sms = 0;
  int rc = device_info(&sms);
  if (rc != QMOE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the route zeroes the error word itself
  return cuda_rc(launch_route(topk_ids_dev, M * top_k, E, tile_n, offsets_dev, sorted_pair_dev,
                              pair_pos_dev, tiles_dev, n_tiles_dev,
                              reinterpret_cast<unsigned int*>(workspace_dev),
                              reinterpret_cast<uint8_t*>(workspace_dev) + kWsHeaderBytes, s));
}

size_t qmoe_repacked_fp4_size(int E, int N, int K) {
  if (E < 1 || N < 1 || K < 1) return 0;
  return (size_t)E * N * (K / 2);
}

size_t qmoe_repacked_scale_size(int E, int N, int K) {
  if (E < 1 || N < 1 || K < 1) return 0;
  return (size_t)E * N * (K / 16);
}

int moe_nvfp4_repack_layout(const uint8_t* w_fp4_dev, const uint8_t* w_scale_dev, int E, int N,
                            int K, int which, int scale_layout, uint8_t* out_fp4_dev,
                            uint8_t* out_scale_dev, void* stream) {
  if (which != QMOE_W13 && which != QMOE_W2) return QMOE_ERR_ARG;
  if (scale_layout != QMOE_SCALES_PLAIN && scale_layout != QMOE_SCALES_SWIZZLED_128X4 &&
      scale_layout != QMOE_SCALES_PACKED_U32)
    return QMOE_ERR_ARG;
  if (E < 1 || E > 2048 || N < 128 || K < 128 || N % 128 || K % 128 || N > 131072 || K > 65536)
    return QMOE_ERR_SHAPE;
  if (!w_fp4_dev || !w_scale_dev || !out_fp4_dev || !out_scale_dev) return QMOE_ERR_ARG;
  if (((uintptr_t)w_fp4_dev | (uintptr_t)w_scale_dev | (uintptr_t)out_fp4_dev |
       (uintptr_t)out_scale_dev) & 15)
    return QMOE_ERR_ARG;
  int sms = 0;
  int rc = device_info(&sms);
  if (rc != QMOE_OK) return rc;
  return cuda_rc(launch_repack(w_fp4_dev, w_scale_dev, E, N, K, which == QMOE_W13, scale_layout,
                               out_fp4_dev, out_scale_dev, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_nvfp4_repack(const uint8_t* w_fp4_dev, const uint8_t* w_scale_dev, int E, int N, int K,
                     int which, uint8_t* out_fp4_dev, uint8_t* out_scale_dev, void* stream) {
  return moe_nvfp4_repack_layout(w_fp4_dev, w_scale_dev, E, N, K, which, QMOE_SCALES_PLAIN,
                                 out_fp4_dev, out_scale_dev, stream);
}

size_t qmoe_forward_workspace_size(int M, int H, int I, int E, int top_k, int sched) {
  if (check_shape(M, H, I, E, top_k) != QMOE_OK) return 0;
  return forward_layout(M, H, I, E, top_k, sched).total;
}

static int forward_impl(const void* x_dev, const uint8_t* w13_fp4_dev, const uint8_t* w13_scale_dev,
                        const float* w13_gscale_dev, const uint8_t* w2_fp4_dev,
                        const uint8_t* w2_scale_dev, const float* w2_gscale_dev,
                        const int32_t* topk_ids_dev, const float* topk_weights_dev, void* out_dev,
                        int M, int H, int I, int E, int top_k, int sched, void* workspace_dev,
                        size_t ws_bytes, void* stream, void* const* events,
                        float swiglu_limit = INFINITY) {
  int rc = check_shape(M, H, I, E, top_k);
  if (rc != QMOE_OK) return rc;
  if (sched < QMOE_SCHED_AUTO || sched > QMOE_SCHED_PREFILL_PAIR) return QMOE_ERR_ARG;
  if (!(swiglu_limit > 0.0f)) return QMOE_ERR_ARG;  // also NaN
  if (M == 0) return QMOE_OK;
  if (!x_dev || !w13_fp4_dev || !w13_scale_dev || !w13_gscale_dev || !w2_fp4_dev ||
      !w2_scale_dev || !w2_gscale_dev || !topk_ids_dev || !topk_weights_dev || !out_dev ||
      !workspace_dev)
    return QMOE_ERR_ARG;
  if (((uintptr_t)x_dev | (uintptr_t)out_dev | (uintptr_t)w13_fp4_dev | (uintptr_t)w13_scale_dev |
       (uintptr_t)w2_fp4_dev | (uintptr_t)w2_scale_dev) & 15)
    return QMOE_ERR_ARG;
  if ((uintptr_t)workspace_dev & 255) return QMOE_ERR_ARG;
  const ForwardLayout L = forward_layout(M, H, I, E, top_k, sched);
  if (ws_bytes < L.total) return QMOE_ERR_WORKSPACE;
  int sms = 0;
  rc = device_info(&sms);
  if (rc != QMOE_OK) return rc;
  const int rsched = resolve_sched(sched, M, top_k, E);
  const int P = M * top_k;
  {
    // the GEMMs count a CTA's K steps (decode pipeline: all units' steps) in 32 bits
    const bool all_steps = rsched == QMOE_SCHED_DECODE || rsched == kSchedPrefillNarrow;
    const unsigned long long steps_cap = all_steps ? (1ull << 31) : (unsigned long long)sms << 31;
    const unsigned long long k1 = H / 128, k2 = I / 128;
    if ((unsigned long long)L.max_tiles * (2 * I / 128) * k1 >= steps_cap ||
        (unsigned long long)L.max_tiles * (H / 128) * k2 >= steps_cap)
      return QMOE_ERR_SHAPE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace_dev);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* sorted_pair = reinterpret_cast<int32_t*>(ws + L.sorted_pair);
  int32_t* pair_pos = reinterpret_cast<int32_t*>(ws + L.pair_pos);
  int32_t* tiles = reinterpret_cast<int32_t*>(ws + L.tiles);
  int32_t* n_tiles = reinterpret_cast<int32_t*>(ws + L.n_tiles);
  void* xs = ws + L.xs;
  void* h = ws + L.h;
  float* ypart = reinterpret_cast<float*>(ws + L.ypart);

  CUtensorMap map_x, map_h;
  const int box_rows = gemm_b_box_rows(rsched), box_slabs = gemm_b_box_slabs(rsched);
  if (make_tmap_rows(&map_x, xs, L.rows, H, box_rows, box_slabs) != QMOE_OK) return QMOE_ERR_CUDA;
  if (make_tmap_rows(&map_h, h, L.rows, I, box_rows, box_slabs) != QMOE_OK) return QMOE_ERR_CUDA;
  // split prefill schedule: the small tiles' launches read 3-D boxes of 64 rows
  const bool split = rsched == kSchedPrefillNarrow;
  int32_t* tile_order = split ? reinterpret_cast<int32_t*>(ws + L.tile_order) : nullptr;
  CUtensorMap map_xs, map_hs;
  if (split) {
    const int br = gemm_b_box_rows(kSchedPrefillSmall), bs = gemm_b_box_slabs(kSchedPrefillSmall);
    if (make_tmap_rows(&map_xs, xs, L.rows, H, br, bs) != QMOE_OK) return QMOE_ERR_CUDA;
    if (make_tmap_rows(&map_hs, h, L.rows, I, br, bs) != QMOE_OK) return QMOE_ERR_CUDA;
  }

  auto mark = [&](int i) -> bool {
    return !events || cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
  };
  // the route zeroes the error word and the split-unit counters itself (and runs as a
  // programmatic dependent of the stream's previous kernel)
  const bool pdl = forward_uses_pdl(rsched);
  if (!mark(0)) return QMOE_ERR_CUDA;
  cudaError_t e = launch_route(topk_ids_dev, P, E, L.tile_n, offsets, sorted_pair, pair_pos, tiles,
                               n_tiles, err, ws + L.route_scratch, s, tile_order, kSmallTileRows,
                               (int)(L.clear_bytes / 4), pdl);
  if (e != cudaSuccess || !mark(1)) return QMOE_ERR_CUDA;
  e = launch_gather(x_dev, pair_pos, M, top_k, H, xs, sms, s, pdl);
  if (e != cudaSuccess || !mark(2)) return QMOE_ERR_CUDA;

  GemmParams p1;
  memset(&p1, 0, sizeof(p1));
  p1.wcodes = w13_fp4_dev;
  p1.wscales = w13_scale_dev;
  p1.gscale = w13_gscale_dev;
  p1.tiles = tiles;
  p1.n_tiles = n_tiles;
  p1.K = H;
  p1.nrb = 2 * I / 128;
  p1.h = h;
  p1.I = I;
  p1.swiglu_limit = swiglu_limit;
  p1.err = err;
  p1.dq_mul[0] = dequant_mul().m64;
  p1.dq_mul[1] = dequant_mul().m4;
  p1.sk_part = reinterpret_cast<float*>(ws + L.sk_part);
  p1.sk_cnt = reinterpret_cast<int*>(ws + L.sk_cnt1);
  p1.tile_order = tile_order;
  p1.tile_part = split ? 1 : 0;
  e = launch_gemm(GemmKind::kFc1, rsched, map_x, p1, sms, s);
  if (e == cudaSuccess && split) {
    p1.tile_part = 2;
    e = launch_gemm(GemmKind::kFc1, kSchedPrefillSmall, map_xs, p1, sms, s);
  }
  if (e != cudaSuccess || !mark(3)) return QMOE_ERR_CUDA;

  GemmParams p2;
  memset(&p2, 0, sizeof(p2));
  p2.wcodes = w2_fp4_dev;
  p2.wscales = w2_scale_dev;
  p2.gscale = w2_gscale_dev;
  p2.tiles = tiles;
  p2.n_tiles = n_tiles;
  p2.K = I;
  p2.nrb = H / 128;
  p2.ypart = ypart;
  p2.sorted_pair = sorted_pair;
  p2.topk_w = topk_weights_dev;
  p2.H = H;
  p2.err = err;
  p2.dq_mul[0] = dequant_mul().m64;
  p2.dq_mul[1] = dequant_mul().m4;
  p2.sk_part = reinterpret_cast<float*>(ws + L.sk_part);
  p2.sk_cnt = reinterpret_cast<int*>(ws + L.sk_cnt2);
  p2.tile_order = tile_order;
  p2.tile_part = split ? 1 : 0;
  e = launch_gemm(GemmKind::kFc2, rsched, map_h, p2, sms, s);
  if (e == cudaSuccess && split) {
    p2.tile_part = 2;
    e = launch_gemm(GemmKind::kFc2, kSchedPrefillSmall, map_hs, p2, sms, s);
  }
  if (e != cudaSuccess || !mark(4)) return QMOE_ERR_CUDA;

  e = launch_combine(ypart, topk_ids_dev, M, top_k, E, H, out_dev, sms, s, pdl);
  if (e != cudaSuccess || !mark(5)) return QMOE_ERR_CUDA;
  return QMOE_OK;
}

int qmoe_forward_workspace_layout(int M, int H, int I, int E, int top_k, int sched,
                                  size_t* layout_out) {
  if (!layout_out) return QMOE_ERR_ARG;
  if (sched < QMOE_SCHED_AUTO || sched > QMOE_SCHED_PREFILL_PAIR) return QMOE_ERR_ARG;
  int rc = check_shape(M, H, I, E, top_k);
  if (rc != QMOE_OK) return rc;
  const ForwardLayout L = forward_layout(M, H, I, E, top_k, sched);
  const size_t v[10] = {L.offsets, L.sorted_pair, L.pair_pos, L.tiles, L.n_tiles,
                        L.xs,      L.h,           L.ypart,    L.total, (size_t)L.rows};
  for (int i = 0; i < 10; ++i) layout_out[i] = v[i];
  return QMOE_OK;
}

int moe_nvfp4_forward(const void* x_dev, const uint8_t* w13_fp4_dev, const uint8_t* w13_scale_dev,
                      const float* w13_gscale_dev, const uint8_t* w2_fp4_dev,
                      const uint8_t* w2_scale_dev, const float* w2_gscale_dev,
                      const int32_t* topk_ids_dev, const float* topk_weights_dev, void* out_dev,
                      int M, int H, int I, int E, int top_k, int sched, void* workspace_dev,
                      size_t ws_bytes, void* stream) {
  return forward_impl(x_dev, w13_fp4_dev, w13_scale_dev, w13_gscale_dev, w2_fp4_dev, w2_scale_dev,
                      w2_gscale_dev, topk_ids_dev, topk_weights_dev, out_dev, M, H, I, E, top_k,
                      sched, workspace_dev, ws_bytes, stream, nullptr);
}

int moe_nvfp4_forward_limit(const void* x_dev, const uint8_t* w13_fp4_dev,
                            const uint8_t* w13_scale_dev, const float* w13_gscale_dev,
                            const uint8_t* w2_fp4_dev, const uint8_t* w2_scale_dev,
                            const float* w2_gscale_dev, const int32_t* topk_ids_dev,
                            const float* topk_weights_dev, void* out_dev, int M, int H, int I,
                            int E, int top_k, int sched, float swiglu_limit, void* workspace_dev,
                            size_t ws_bytes, void* stream) {
  return forward_impl(x_dev, w13_fp4_dev, w13_scale_dev, w13_gscale_dev, w2_fp4_dev, w2_scale_dev,
                      w2_gscale_dev, topk_ids_dev, topk_weights_dev, out_dev, M, H, I, E, top_k,
                      sched, workspace_dev, ws_bytes, stream, nullptr, swiglu_limit);
}

int moe_nvfp4_forward_noalloc(const void* x_dev, const uint8_t* w13_fp4_dev,
                              const uint8_t* w13_scale_dev, const float* w13_gscale_dev,
                              const uint8_t* w2_fp4_dev, const uint8_t* w2_scale_dev,
                              const float* w2_gscale_dev, const int32_t* topk_ids_dev,
                              const float* topk_weights_dev, void* out_dev, int M, int H, int I,
                              int E, int top_k, int sched, void* stream) {
  int rc = check_shape(M, H, I, E, top_k);
  if (rc != QMOE_OK) return rc;
  if (sched < QMOE_SCHED_AUTO || sched > QMOE_SCHED_PREFILL_PAIR) return QMOE_ERR_ARG;
  if (M == 0) return QMOE_OK;
  if (forward_layout(M, H, I, E, top_k, sched).total > (size_t)QMOE_NOALLOC_SCRATCH_BYTES)
    return QMOE_ERR_WORKSPACE;  // this batch needs more scratch than the built-in array
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != QMOE_OK) return rc;
  return forward_impl(x_dev, w13_fp4_dev, w13_scale_dev, w13_gscale_dev, w2_fp4_dev, w2_scale_dev,
                      w2_gscale_dev, topk_ids_dev, topk_weights_dev, out_dev, M, H, I, E, top_k,
                      sched, scratch, (size_t)QMOE_NOALLOC_SCRATCH_BYTES, stream, nullptr);
}

int qmoe_noalloc_read_error(void* stream, uint32_t* flags_out) {
  if (!flags_out) return QMOE_ERR_ARG;
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != QMOE_OK) return rc;
  return qmoe_read_error(scratch, stream, flags_out);
}

int moe_nvfp4_forward_events(const void* x_dev, const uint8_t* w13_fp4_dev,
                             const uint8_t* w13_scale_dev, const float* w13_gscale_dev,
                             const uint8_t* w2_fp4_dev, const uint8_t* w2_scale_dev,
                             const float* w2_gscale_dev, const int32_t* topk_ids_dev,
                             const float* topk_weights_dev, void* out_dev, int M, int H, int I,
                             int E, int top_k, int sched, void* workspace_dev, size_t ws_bytes,
                             void* stream, void* const* events) {
  if (!events) return QMOE_ERR_ARG;
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return QMOE_ERR_ARG;
  return forward_impl(x_dev, w13_fp4_dev, w13_scale_dev, w13_gscale_dev, w2_fp4_dev, w2_scale_dev,
                      w2_gscale_dev, topk_ids_dev, topk_weights_dev, out_dev, M, H, I, E, top_k,
                      sched, workspace_dev, ws_bytes, stream, events);
}

int qmoe_read_error(const void* workspace_dev, void* stream, uint32_t* flags_out) {
  if (!workspace_dev || !flags_out) return QMOE_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t flags = 0;
  if (cudaMemcpyAsync(&flags, workspace_dev, sizeof(flags), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QMOE_ERR_CUDA;
  *flags_out = flags;
  if (flags & QMOE_FLAG_INTERNAL) return QMOE_ERR_CUDA;
  if (flags & QMOE_FLAG_TIMEOUT) return QMOE_ERR_TIMEOUT;
  if (flags & QMOE_FLAG_BAD_ID) return QMOE_ERR_BAD_ID;
  return QMOE_OK;
}

int qmoe_selftest_dequant(uint16_t* out_dev, void* stream) {
  if (!out_dev) return QMOE_ERR_ARG;
  int sms = 0;
  int rc = device_info(&sms);
  if (rc != QMOE_OK) return rc;
  return cuda_rc(launch_selftest_dequant(out_dev, reinterpret_cast<cudaStream_t>(stream)));
}

int qmoe_selftest_timeout(void* workspace_dev, long long limit_ns, void* stream) {
  if (!workspace_dev || limit_ns < 1000 || limit_ns > 1000000000LL) return QMOE_ERR_ARG;
  int sms = 0;
  int rc = device_info(&sms);
  if (rc != QMOE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace_dev, 0, sizeof(unsigned int), s) != cudaSuccess) return QMOE_ERR_CUDA;
  if (launch_selftest_timeout(reinterpret_cast<unsigned int*>(workspace_dev), limit_ns, s) !=
      cudaSuccess)
    return QMOE_ERR_CUDA;
  uint32_t flags = 0;
  return qmoe_read_error(workspace_dev, stream, &flags);
}

}  // extern "C"
