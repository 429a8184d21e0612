/*
 * qmoe — NVFP4 W4A16 mixture-of-experts layer for GB300 (sm_103a).
 *
 * The layer (megamoe_rm.cu page: header comment, route_prep, fc1_rm, fc2_rm,
 * combine; tilelang_kernels.py page: grouped_gemm_fp4):
 *   pairs i = m * top_k + k of M tokens and top_k slots are grouped by expert;
 *   for each pair with expert e:
 *     g   = gs13[e] * x[m] . Wq13[e]^T        (Wq13 [2I][H]: rows 0..I-1 up, I..2I-1 gate)
 *     h   = bf16( SiLU(g[I:2I]) * g[0:I] )
 *     y   = gs2[e] * h . Wq2[e]^T             (Wq2 [H][I])
 *   out[m] = bf16( sum over k ascending of topk_weights[m][k] * y_(m,k) )
 * Wq = E2M1 code * E4M3 block scale (one scale per 16 K-elements of a row); two
 * codes per byte along K, the even K element in the low nibble.  x is bf16.
 *
 * Conventions for every call:
 *  - Pointers named *_dev are device pointers owned by the caller; the library
 *    never allocates, frees or keeps them.  `stream` is a cudaStream_t (may be
 *    NULL for the legacy default stream); all work is enqueued on it and no call
 *    synchronises the host, except qmoe_read_error and qmoe_noalloc_read_error.
 *  - Every call returns QMOE_OK (0) or a negative QMOE_ERR_* code and never
 *    throws or aborts.  Argument checks run before anything is enqueued.
 *  - Shapes: H % 128 == 0, I % 128 == 0, 1 <= E <= 2048, 1 <= top_k <= 64,
 *    M >= 0 (M == 0 is a no-op), M * top_k < 2^31, H, I <= 65536.
 *  - The device must be sm_103 (GB300) or another sm_10x part running sm_103a
 *    code; otherwise QMOE_ERR_ARCH.
 */
#ifndef QMOE_H_
#define QMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMOE_OK 0
#define QMOE_ERR_ARG (-1)       /* null pointer or argument out of range */
#define QMOE_ERR_SHAPE (-2)     /* dimensions violate the shape rules above */
#define QMOE_ERR_CUDA (-3)      /* a CUDA runtime call or launch failed */
#define QMOE_ERR_TIMEOUT (-4)   /* a bounded device-side wait expired (qmoe_read_error) */
#define QMOE_ERR_ARCH (-5)      /* the current device cannot run sm_103a code */
#define QMOE_ERR_WORKSPACE (-6) /* workspace smaller than the size query returned */
#define QMOE_ERR_BAD_ID (-7)    /* an expert id >= E was seen (qmoe_read_error) */

/* Device error-word bits (qmoe_read_error). */
#define QMOE_FLAG_BAD_ID 1u
#define QMOE_FLAG_TIMEOUT 2u
#define QMOE_FLAG_INTERNAL 4u /* a kernel's check of a hardware contract failed */

/* Tile schedules for moe_nvfp4_forward. */
#define QMOE_SCHED_AUTO 0    /* DECODE when M * top_k <= 4 * E, else PREFILL */
#define QMOE_SCHED_DECODE 1  /* tiles of <= 16 pairs: weight streaming, HBM bound */
/* Tensor bound: tiles of <= 320 pairs when experts average >= 192 pairs; else tiles of
   <= 192 pairs, with FC1 and FC2 each run as two launches: the tiles of more than 64
   pairs (whose epilogue overlaps the next tile's MMAs), then the others on the decode
   pipeline. */
#define QMOE_SCHED_PREFILL 2
/* As PREFILL, with each 256-row weight tile on a pair of SMs (tcgen05 2-CTA MMAs, each
   SM holding half of the tile's pair rows); a GEMM whose count of 128-row weight blocks
   is odd runs as PREFILL.  Same results as PREFILL; slower than it at present. */
#define QMOE_SCHED_PREFILL_PAIR 3

/* Weight roles for moe_nvfp4_repack. */
#define QMOE_W13 1 /* w13 [E][2I][H/2]: up and gate rows, interleaved for the SwiGLU epilogue */
#define QMOE_W2 2  /* w2  [E][H][I/2] */

/* Pair-tile height used by each schedule (the moe_route tile_n it runs with). */
int qmoe_sched_tile_n(int sched, int M, int top_k, int E);

/* Upper bound on the number of tiles moe_route can emit: ceil(M*top_k/tile_n) + E. */
int qmoe_max_tiles(int M, int top_k, int E, int tile_n);

/*
 * moe_route — group the M*top_k (token, expert) pairs by expert.
 * Defined by route_prep on the megamoe_rm.cu page (a pair's slot is its rank among
 * earlier pairs with the same expert; expert -1 is skipped) and by the per-expert
 * row offsets of cutlass discussion 2855 ("total tokens including expert").
 *   topk_ids_dev     int32 [M][top_k], row-major; pair i = m * top_k + k.  Ids < 0
 *                    are skipped; ids >= E are skipped and set QMOE_FLAG_BAD_ID in
 *                    the error word (first 4 bytes of `workspace_dev`).
 *   offsets_dev      int32 [E+1]: offsets[e] = valid pairs with expert < e.
 *   sorted_pair_dev  int32 [M*top_k]: pairs in (expert, pair index) order; entries
 *                    at positions >= offsets[E] are -1.
 *   pair_pos_dev     int32 [M*top_k]: inverse of sorted_pair, -1 for skipped pairs.
 *   tiles_dev        int32 [qmoe_max_tiles(...)][3]: (expert, start position, rows),
 *                    rows <= tile_n, experts ascending, positions ascending; only
 *                    the first *n_tiles entries are written.
 *   n_tiles_dev      int32 [1].
 *   workspace_dev    >= qmoe_route_workspace_size(...) bytes, 256-byte aligned; its
 *                    first 4 bytes are the error word, which this call clears first;
 *                    above 8192 pairs it also holds per-warp count tables.
 * The result is bit-exact and deterministic.
 */
size_t qmoe_route_workspace_size(int M, int top_k, int E, int tile_n);
int moe_route(const int32_t* topk_ids_dev, int M, int top_k, int E, int tile_n,
              int32_t* offsets_dev, int32_t* sorted_pair_dev, int32_t* pair_pos_dev,
              int32_t* tiles_dev, int32_t* n_tiles_dev, void* workspace_dev, size_t ws_bytes,
              void* stream);

/*
 * moe_nvfp4_repack — one-time reordering of plain NVFP4 weights into the layout
 * the grouped GEMM streams (a kernel-chosen layout; bytes are only permuted, the
 * sizes equal the inputs').  The principle follows cutlass issue 2087: store the
 * scales in the order the loader consumes them, so tile loads are contiguous.
 *   w_fp4_dev    uint8 [E][N][K/2]  plain codes (low nibble = even k)
 *   w_scale_dev  uint8 [E][N][K/16] plain E4M3 block scales
 *   which        QMOE_W13 (N = 2I, K = H) or QMOE_W2 (N = H, K = I)
 *   out_fp4_dev  uint8, qmoe_repacked_fp4_size(E, N, K) bytes
 *   out_scale_dev uint8, qmoe_repacked_scale_size(E, N, K) bytes
 * N % 128 == 0 and K % 128 == 0 are required (QMOE_ERR_SHAPE otherwise).
 */
/*
 * moe_nvfp4_repack_layout — moe_nvfp4_repack taking the block scales in one of three
 * layouts (output identical for the same scale values):
 *   QMOE_SCALES_PLAIN          [E][N][K/16], row-major (as moe_nvfp4_repack)
 *   QMOE_SCALES_SWIZZLED_128X4 per expert N*K/16 bytes in the 128x4 swizzle that
 *       CUTLASS / FlashInfer NVFP4 checkpoints keep (megamoe_rm.cu page, scale_off):
 *       tiles of 128 rows x 4 scales, 512 bytes each, the 4-column tile index
 *       fastest; inside a tile the scale of row r, column c at
 *       (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4.
 *   QMOE_SCALES_PACKED_U32     uint32 [E][N][K/64], four UE4M3 scales per word
 *       (tilelang_kernels.py page, grouped_gemm_fp4_packed_sf): the scale of K block
 *       4g + j in bits 8j..8j+7 of word g (the page gives no byte order; this is the
 *       order of a little-endian uint32 view of the plain bytes).  w_scale_dev must be
 *       4-byte aligned (16-byte, as for every pointer here).
 * Other arguments and errors as moe_nvfp4_repack; an unknown layout: QMOE_ERR_ARG.
 */
#define QMOE_SCALES_PLAIN 0
#define QMOE_SCALES_SWIZZLED_128X4 1
#define QMOE_SCALES_PACKED_U32 2
int moe_nvfp4_repack_layout(const uint8_t* w_fp4_dev, const uint8_t* w_scale_dev, int E, int N,
                            int K, int which, int scale_layout, uint8_t* out_fp4_dev,
                            uint8_t* out_scale_dev, void* stream);

size_t qmoe_repacked_fp4_size(int E, int N, int K);
size_t qmoe_repacked_scale_size(int E, int N, int K);
int moe_nvfp4_repack(const uint8_t* w_fp4_dev, const uint8_t* w_scale_dev, int E, int N, int K,
                     int which, uint8_t* out_fp4_dev, uint8_t* out_scale_dev, void* stream);

/*
 * moe_nvfp4_forward — the whole layer: route, gather, grouped FC1 + SwiGLU, grouped
 * FC2, weighted top_k combine.  Follows megamoe_rm_forward on the megamoe_rm.cu
 * page (scratch passed in by the caller, work on the caller's stream, shape
 * checks up front).
 *   x_dev           bf16 [M][H]
 *   w13_fp4_dev, w13_scale_dev   repacked w13 (moe_nvfp4_repack with QMOE_W13)
 *   w13_gscale_dev  fp32 [E], multiplies the FC1 accumulator
 *   w2_fp4_dev, w2_scale_dev     repacked w2 (moe_nvfp4_repack with QMOE_W2)
 *   w2_gscale_dev   fp32 [E], multiplies the FC2 accumulator
 *   topk_ids_dev    int32 [M][top_k]  (ids < 0 skipped, ids >= E flagged and skipped)
 *   topk_weights_dev fp32 [M][top_k], used as given
 *   out_dev         bf16 [M][H]
 *   sched           QMOE_SCHED_*
 *   workspace_dev   >= qmoe_forward_workspace_size(M, H, I, E, top_k, sched) bytes,
 *                   256-byte aligned; holds the error word, routing tables, the
 *                   gathered activations, h and the per-pair partial outputs.  Its
 *                   contents on entry do not matter: the call zeroes what it needs
 *                   (the error word and the decode schedule's counters) itself.
 * Deterministic: two calls on the same inputs give bitwise equal outputs.  Calls
 * sharing one workspace must not overlap on the GPU.
 */
size_t qmoe_forward_workspace_size(int M, int H, int I, int E, int top_k, int sched);
/* Kernels one moe_nvfp4_forward call launches (route, gather, FC1, FC2, combine; the
 * route is three kernels above 8192 pairs, and FC1 and FC2 are two launches each on the
 * prefill schedule when experts average fewer than 192 pairs); 0 for M = 0,
 * QMOE_ERR_ARG for bad sizes. */
int qmoe_forward_kernel_count(int M, int top_k, int E, int sched);
int moe_nvfp4_forward(const void* x_dev, const uint8_t* w13_fp4_dev, const uint8_t* w13_scale_dev,
                      const float* w13_gscale_dev, const uint8_t* w2_fp4_dev,
                      const uint8_t* w2_scale_dev, const float* w2_gscale_dev,
                      const int32_t* topk_ids_dev, const float* topk_weights_dev, void* out_dev,
                      int M, int H, int I, int E, int top_k, int sched, void* workspace_dev,
                      size_t ws_bytes, void* stream);

/*
 * moe_nvfp4_forward_limit — moe_nvfp4_forward with the GLM form of the SwiGLU
 * (megamoe_rm.cu page, fc1_rm epilogue): before h = bf16(SiLU(gate) * up), gate is
 * clamped from above and up to [-swiglu_limit, swiglu_limit].
 *   swiglu_limit  > 0; +infinity gives exactly moe_nvfp4_forward's results; zero,
 *                 negative or NaN: QMOE_ERR_ARG.
 * Other arguments, results and errors as moe_nvfp4_forward.  With a finite limit
 * QMOE_SCHED_PREFILL_PAIR runs as QMOE_SCHED_PREFILL.
 */
int moe_nvfp4_forward_limit(const void* x_dev, const uint8_t* w13_fp4_dev,
                            const uint8_t* w13_scale_dev, const float* w13_gscale_dev,
                            const uint8_t* w2_fp4_dev, const uint8_t* w2_scale_dev,
                            const float* w2_gscale_dev, const int32_t* topk_ids_dev,
                            const float* topk_weights_dev, void* out_dev, int M, int H, int I,
                            int E, int top_k, int sched, float swiglu_limit, void* workspace_dev,
                            size_t ws_bytes, void* stream);

/*
 * moe_nvfp4_forward_noalloc — moe_nvfp4_forward for callers that cannot allocate
 * device memory: a plugin called from inside another runtime's enqueue step with no
 * allocator handed to it, a C host program that does not own the process's memory
 * pool, or a serving loop that must not allocate once it is running.  It takes the
 * same inputs and outputs (all still passed in by the caller) but no workspace:
 * it uses a scratch array of QMOE_NOALLOC_SCRATCH_BYTES (16 MiB) built into the
 * library, which every GPU that loads the library holds until the process exits.
 *  - Size limit: the batch must fit that array, i.e. qmoe_forward_workspace_size(
 *    M, H, I, E, top_k, sched) <= QMOE_NOALLOC_SCRATCH_BYTES (decode-sized batches:
 *    e.g. M = 16, H = 7168, I = 2048, top_k = 8 needs about 9 MB); larger batches get
 *    QMOE_ERR_WORKSPACE before anything is enqueued.
 *  - Set-up: the array's device address is looked up (cudaGetSymbolAddress) on the
 *    first call made on a device, and again whenever a call finds another CUDA context
 *    current than the one of the last lookup (after cudaDeviceReset, or when the caller
 *    runs its own context); it is the address in the context current at the call.  A
 *    lookup makes the device's primary context current if the thread had none.  Make
 *    the first call on a device, and the first call in a new context, before any stream
 *    capture.  The lookup is guarded by a lock, so threads may make first calls at once.
 *  - It calls no cudaMalloc / cudaFree and no allocating library routine.
 *  - Every call shares the one array and leaves its contents behind; the error word
 *    in it is cleared at the start of each call.  Calls that overlap on the GPU (on
 *    different streams, or from several host threads) race on the array and give
 *    wrong results: serialise them.  qmoe_noalloc_read_error reads the error word
 *    (bad expert ids, expired waits) of the last call.
 * The pages have no counterpart of this entry point.
 */
#define QMOE_NOALLOC_SCRATCH_BYTES (16u << 20)
int moe_nvfp4_forward_noalloc(const void* x_dev, const uint8_t* w13_fp4_dev,
                              const uint8_t* w13_scale_dev, const float* w13_gscale_dev,
                              const uint8_t* w2_fp4_dev, const uint8_t* w2_scale_dev,
                              const float* w2_gscale_dev, const int32_t* topk_ids_dev,
                              const float* topk_weights_dev, void* out_dev, int M, int H, int I,
                              int E, int top_k, int sched, void* stream);

/*
 * qmoe_noalloc_read_error — qmoe_read_error for moe_nvfp4_forward_noalloc: copies the
 * error word of the built-in scratch array (current device and context) to the host
 * after the stream's work so far; synchronises `stream`.  Same flags and return codes
 * as qmoe_read_error.  (No counterpart on the pages.)
 */
int qmoe_noalloc_read_error(void* stream, uint32_t* flags_out);

/*
 * qmoe_forward_workspace_layout — byte offsets, inside a forward workspace, of what
 * moe_nvfp4_forward leaves there, for inspection by tests and tools:
 *   layout_out[0] offsets [E+1] int32      [1] sorted_pair [M*top_k] int32
 *   layout_out[2] pair_pos [M*top_k] int32 [3] tiles [max_tiles][3] int32
 *   layout_out[4] n_tiles int32            [5] xs: gathered x rows [rows][H] bf16
 *   layout_out[6] h [rows][I] bf16, row = a pair's sorted position
 *   layout_out[7] ypart [M*top_k][H] fp32, row = pair index
 *   layout_out[8] total bytes              [9] rows (M*top_k rounded up to 16)
 * layout_out must hold 10 entries.  (An inspection aid; no counterpart on the pages.)
 */
int qmoe_forward_workspace_layout(int M, int H, int I, int E, int top_k, int sched,
                                  size_t* layout_out);

/*
 * moe_nvfp4_forward_events — moe_nvfp4_forward that also records six caller-owned
 * cudaEvent_t at its stage boundaries on `stream`, so that each kernel can be timed
 * on the stream it runs on: events[0] before route, [1] after route, [2] after the
 * activation gather, [3] after FC1, [4] after FC2, [5] after combine.  Same
 * arguments, results and errors as moe_nvfp4_forward; QMOE_ERR_ARG if `events` or
 * any of its six entries is NULL.  (A measurement hook; no counterpart on the pages.)
 */
int moe_nvfp4_forward_events(const void* x_dev, const uint8_t* w13_fp4_dev,
                             const uint8_t* w13_scale_dev, const float* w13_gscale_dev,
                             const uint8_t* w2_fp4_dev, const uint8_t* w2_scale_dev,
                             const float* w2_gscale_dev, const int32_t* topk_ids_dev,
                             const float* topk_weights_dev, void* out_dev, int M, int H, int I,
                             int E, int top_k, int sched, void* workspace_dev, size_t ws_bytes,
                             void* stream, void* const* events);

/*
 * qmoe_read_error — copy the device error word (first 4 bytes of a route or forward
 * workspace) to the host after the stream's work so far; synchronises `stream`.
 * *flags_out gets the QMOE_FLAG_* bits.  Returns QMOE_ERR_CUDA if the internal bit
 * is set (the layer's results are not valid), else QMOE_ERR_TIMEOUT if the timeout
 * bit is set, else QMOE_ERR_BAD_ID if the bad-id bit is set, else QMOE_OK.
 */
int qmoe_read_error(const void* workspace_dev, void* stream, uint32_t* flags_out);

/*
 * Diagnostics used by the tests (no counterpart on the pages).
 * qmoe_selftest_dequant: dequantizes, for every c (0..15) and E4M3 scale byte s
 *   (0..255), one packed word holding the E2M1 codes (c + j) mod 16 at its element
 *   positions j = 0..7 with scale s, and writes the bf16 of code * scale of position j
 *   to out_dev[(c * 256 + s) * 8 + j] (uint16 bf16 bits, 32768 entries, 64 KB).
 *   Every product is exact.
 * qmoe_selftest_timeout: runs the bounded mbarrier wait of the GEMM kernels on a
 *   barrier nothing arrives at, with a limit of `limit_ns` nanoseconds, and records
 *   the expiry in the error word at workspace_dev (>= 256 bytes).  Returns
 *   QMOE_ERR_TIMEOUT when the wait expired as it must, QMOE_OK otherwise.
 */
int qmoe_selftest_dequant(uint16_t* out_dev, void* stream);
int qmoe_selftest_timeout(void* workspace_dev, long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H_ */
