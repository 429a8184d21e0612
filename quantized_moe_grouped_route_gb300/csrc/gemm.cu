// Persistent grouped GEMM for FC1 (+ SwiGLU) and FC2 (+ global scale and routing
// weight) of the NVFP4 W4A16 MoE layer, on tcgen05 tensor cores.
//
// What it computes (megamoe_rm.cu page, fc1_rm / fc2_rm):
//   FC1 tile (expert e, 128 weight rows rb, pair tile t):
//     g = gs13[e] * Wq13[e][rows] . xs[t]^T, then h = bf16(SiLU(gate) * up), with
//     the GLM clamp of gate and up first when a SwiGLU limit is given (CLAMP)
//   FC2 tile: y = gs2[e] * Wq2[e][rows] . h[t]^T, ypart[pair][j] = topk_w[pair] * y
// Each unit is one 128-row block of one expert's weights against one tile of that
// expert's pairs (<= NMAX pairs) over the whole K: the weights are the MMA's M side
// ("swap AB": weight rows on M = 128, pairs on N = 16..256; a wider tile as two
// MMAs per K slice), so small per-expert batches still fill the instruction.  Every
// output element is summed in a fixed order: by one CTA, or (decode pipeline, 16-pair
// tiles) from the K-ordered partial sums of the CTAs a unit was split between
// (sk_reduce), so results are deterministic.  A launch covers all tiles or one part
// of the split prefill schedule's tile order (GemmParams::tile_part).
//
// Data path per pipeline step (KS x 128 of K):
//   weight TMA    : bulk copies of the step's packed codes (8 KB per block) and scales
//                   (1 KB per block) into the weight ring
//   pair rows     : tiled TMA of the tile's gathered activations (bf16, 128-byte
//                   swizzle) into the slot's shared-memory stage, from a producer warp
//                   or (decode, 16-pair tiles) the MMA warps
//   dequant warps : codes -> bf16 in registers (bit placement + one bf16x2 multiply
//                   by the block scale) -> tcgen05.st into TMEM (the MMA's A operand)
//   MMA warp(s)   : 8 x tcgen05.mma kind::f16 per block, A from TMEM, B from smem,
//                   fp32 accumulator in TMEM; commits release the slot
//   epilogue warps: tcgen05.ld of the accumulator, scale, SwiGLU or routing weight,
//                   global stores
// The dequantized weights never touch shared memory, which leaves the smem
// bandwidth to TMA and the MMA's B reads.
//
// Every wait is bounded (qmoe::mbar_wait): on expiry the CTA raises the timeout bit
// in the error word, the roles leave their loops, in-flight copies and MMAs are
// drained with bounded waits, and TMEM is released before the CTA exits.
#include <cmath>

#include "common.cuh"
#include "dequant.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace qmoe {
namespace {

constexpr int kBK = 128;            // K per weight block of the repacked layout
constexpr int kCodeBytes = 8192;    // 128 rows x 128 K / 2
constexpr int kScaleBytes = 1024;   // 128 rows x 8 blocks
constexpr int kRawBytes = kCodeBytes + kScaleBytes;
constexpr int kTmemCols = 512;
constexpr int kCtrlBytes = 1024;    // barriers, TMEM slot, abort flag

// Warp roles: 1..NMW MMA issue (NMW <= 3), 4..7 epilogue (one per TMEM lane quarter),
// 8.. dequant (DG groups of 4 warps); with BIN the MMA warps also issue the pair-row
// copies of their own steps and warp 0 is the weight TMA producer, otherwise warp 0
// is a pair-row TMA producer and warp 2 the weight producer.  Warp w runs on scheduler
// w % 4 and may only touch TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31, so every group of
// four consecutive warps covers the 128 lanes once.  Each scheduler carries one dequant
// warp per group; the per-step control work (eight tcgen05.mma, costly to issue next
// to busy dequant warps, the pair-row copy and the weight copies) is spread so that no
// scheduler carries much more of it than the others.
constexpr int kMmaWarp0 = 1;
constexpr int kEpiWarp0 = 4;
constexpr int kPairBoxRows = 64;  // rows of a 2-D pair-row box (prefill schedule)
constexpr int kDequantWarp0 = 8;
__host__ __device__ constexpr int weight_tma_warp(bool bin) { return bin ? 0 : 2; }
__host__ __device__ constexpr int pair_tma_warp(bool bin) { return bin ? -1 : 0; }
__host__ __device__ constexpr int gemm_threads(int groups) { return (kDequantWarp0 + 4 * groups) * 32; }

// Two rings:
//   raw ring (RS stages): packed codes + scales of one 128-wide K step, refilled as
//            soon as the dequant warps have read it, so many weight bytes stay in
//            flight per SM (the decode bound is HBM latency x bandwidth);
//   slots    (SL): one K step's operands for the MMA: the dequantized bf16 weights in
//            a 64-column TMEM slot and the tile's pair rows in an smem stage.  A slot
//            is "full" when its 4 dequant warps have arrived and the pair rows have
//            landed, and "empty" when the MMAs that read it have completed.
// MMA issue: NMW warps take the K steps round robin by global step index, each into
// its own accumulator; the epilogue adds the accumulators in a fixed order, so the
// result does not depend on timing.
// Barrier waits use phase parity, which cannot tell phase k from phase k+2.  Every
// slot must therefore be filled and drained by single ordered streams: all uses of a
// slot (steps s, s+SL, s+2SL, ..) go to the same dequant group and the same MMA warp,
// i.e. SL is a multiple of DG and of NMW, and likewise RS of DG for the weight ring.
// Otherwise a warp that runs a full ring cycle ahead of asynchronous completions
// (which may land out of order) can pass a wait early, and the rings desynchronise
// (checked by simulating the protocol).
//
// Pair rows: with BIN the tile's rows of one K step (both 64-wide slabs) arrive in a
// single 3-D box copy {64 elements, NMAX rows, 2 slabs}, issued by the MMA warp that
// owns the step; otherwise a producer warp copies 2-D boxes of kPairBoxRows rows x 64
// elements, as many as the tile needs, slab by slab: a slot's slab 0 is refilled as
// soon as the MMAs of the previous step that read it have completed (their own
// commit), and slab 1 lands on its own barrier, which gives the copies (up to 80 KB a
// step, more time than the step's MMAs take at the rate the pair rows arrive) half a
// step more lead than whole-slot refills.  One copy per step, from warps spread over
// the schedulers, keeps copy issue off the path that feeds the MMA.
// A pipeline step covers KS weight blocks (KS x 128 of K): KS x 9 KB of the weight ring,
// a TMEM A slot of KS x 64 columns, 2 KS slabs of pair rows and 8 KS MMAs, so the
// per-step barrier and bookkeeping work is paid once per KS blocks.  The last step of
// a unit covers the remaining nb128 - (nss - 1) KS blocks ("halves").
template <int NMAX, int RS, int SL, int ACCB, int DG, int NMW, int KS>
struct Cfg {
  static constexpr int kBSlab = NMAX * 128;  // one 64-wide K slab of B: NMAX rows x 128 bytes
  static constexpr int kBBytes = 2 * KS * kBSlab;
  static constexpr int kStageBytes = KS * kRawBytes;  // [KS codes blocks][KS scale blocks]
  static constexpr int kSlotCols = 64 * KS;
  static constexpr int kAccCol0 = SL * kSlotCols;  // TMEM: [A slots][acc: ACCB x NMW x NMAX]
  // epilogue staging on the prefill schedule, per epilogue warp: a tile's pair ids and
  // weights (FC2) or a 512-byte transpose tile (FC1)
  static constexpr int kEpiBytes = NMW == 1 ? 4 * NMAX * 8 : 0;
  static constexpr int kSmemBytes = SL * kBBytes + RS * kStageBytes + 1024 + kCtrlBytes + kEpiBytes;
  static constexpr int kThreads = gemm_threads(DG);
  static_assert(KS == 1 || KS == 2, "weight blocks per step");
  static_assert(kBBytes % 1024 == 0 && kStageBytes % 1024 == 0, "1024-byte stage alignment");
  static_assert(SL * kSlotCols + ACCB * NMW * NMAX <= kTmemCols, "TMEM budget");
  // a tile wider than one MMA's N (256) takes two accumulator chains (256 + the rest)
  static_assert(NMAX % 16 == 0 && NMAX >= 16 && (NMAX <= 256 || (NMAX <= 512 && NMW == 1)),
                "MMA N range");
  static_assert(NMW >= 1 && NMW <= 3, "MMA warps 1..3");
  static_assert(SL % DG == 0 && SL % NMW == 0, "each slot needs one dequant group and one MMA warp");
  static_assert(RS % DG == 0, "each weight stage needs one dequant group");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert((2 * RS + SL * (KS + 3) + 2 * ACCB + 1) * 8 + 16 <= 1024, "barrier area");
};

// Stream-K ranges of the decode schedule: CTA c of G takes the global steps
// [sk_range_start(c), sk_range_start(c + 1)) of the n_steps steps of all units.
__host__ __device__ __forceinline__ uint32_t sk_range_start(unsigned long long n_steps,
                                                           unsigned int c, unsigned int G) {
  return (uint32_t)(n_steps * c / G);
}
// Whether the decode schedule splits units between CTAs: only when dealing whole units
// (ceil(n_units / G) per CTA at most) would leave more than two K steps per CTA idle on
// average; below that the partial sums cost more than the balance gains (measured:
// splitting gained 2% on FC1 of the M = 16 decode workload, 21.7 units of 28 steps per
// CTA, and lost 10% on FC2 of the M = 1 one, 2.95 units of 12 steps).
__host__ __device__ __forceinline__ bool sk_split(long long n_units, int nks, unsigned int G) {
  const long long waves = (n_units + G - 1) / G;
  return (waves * (long long)G - n_units) * nks > 2LL * G;
}
// The CTA whose range holds global step g: the largest c with sk_range_start(c) <= g,
// i.e. ceil((g + 1) G / n_steps) - 1.
__host__ __device__ __forceinline__ unsigned int sk_cta_of(unsigned long long g,
                                                          unsigned long long n_steps,
                                                          unsigned int G) {
  return (unsigned int)(((g + 1) * G + n_steps - 1) / n_steps - 1);
}

// Decode schedule, a unit split between CTAs: each segment's epilogue warp q stores its
// 32 rows x 16 pairs of partial sums (fp32) in the CTA's slot (0 when the unit is the
// CTA's first, else 1), then counts itself in the unit's arrival counter for quarter q.
// The warp that arrives last sums all segments' partials in K order (CTA order), its own
// from registers, the others' from global memory, into v and returns true; the others
// return false.  The sum order does not depend on which segment arrives last, so the
// result is deterministic; no warp waits for another.
__device__ __forceinline__ bool sk_reduce(const GemmParams& p, float (&v)[16], int u, int nks,
                                          unsigned long long n_steps, uint32_t g0, int lane,
                                          int q) {
  const unsigned int G = gridDim.x;
  const int row = q * 32 + lane;
  const unsigned long long first = (unsigned long long)u * nks, last = first + nks - 1;
  const unsigned int c0 = sk_cta_of(first, n_steps, G), c1 = sk_cta_of(last, n_steps, G);
  int nseg = 0;
  for (unsigned int c = c0; c <= c1; ++c)
    nseg += sk_range_start(n_steps, c + 1, G) > sk_range_start(n_steps, c, G);
  // one counter per (split unit, lane quarter), indexed by the CTA that holds the unit's
  // first step: a CTA's range starts at most one unit that runs past its end
  int* cnt = p.sk_cnt + (size_t)c0 * 4 + q;
  // Every other segment already counted (the usual case for a CTA's last segment, whose
  // unit the next CTA began at its start): this warp is the last one, and no other warp
  // can see that count without having counted itself first.  Its own partial then needs
  // no store, fence or count; each lane's acquire load orders its reads of the others'
  // partials after their stores.
  int seen;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(cnt) : "memory");
  if (__all_sync(0xffffffffu, seen == nseg - 1)) {
    // (falls through to the sum below)
  } else {
    const int slot = (int)(g0 / (uint32_t)nks) == u ? 0 : 1;
    float4* mine =
        reinterpret_cast<float4*>(p.sk_part + ((size_t)(blockIdx.x * 2 + slot) * 128 + row) * 16);
#pragma unroll
    for (int c = 0; c < 4; ++c) mine[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(cnt, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != nseg - 1) return false;
    __threadfence();
  }
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;
  for (unsigned int c = c0; c <= c1; ++c) {
    const uint32_t cs = sk_range_start(n_steps, c, G);
    if (sk_range_start(n_steps, c + 1, G) == cs) continue;  // an empty range
    if (c == blockIdx.x) {
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] += v[k];
    } else {
      const int sc = (int)(cs / (uint32_t)nks) == u ? 0 : 1;
      const float4* src =
          reinterpret_cast<const float4*>(p.sk_part + ((size_t)(c * 2 + sc) * 128 + row) * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 w = __ldcg(src + k);
        acc[4 * k] += w.x;
        acc[4 * k + 1] += w.y;
        acc[4 * k + 2] += w.z;
        acc[4 * k + 3] += w.w;
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = acc[c];
  return true;
}

// The units of a launch: each tile of its part (GemmParams::tile_part) times the p.nrb
// weight row blocks, unit u = j * nrb + rb for the part's j-th tile.
__device__ __forceinline__ int part_tiles(const GemmParams& p) {
  if (p.tile_part == 0) return p.n_tiles[0];
  return p.tile_part == 1 ? p.n_tiles[1] : p.n_tiles[0] - p.n_tiles[1];
}
__device__ __forceinline__ int part_tile(const GemmParams& p, int j) {
  if (p.tile_part == 0) return j;
  return p.tile_order[(p.tile_part == 1 ? 0 : p.n_tiles[1]) + j];
}

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer_ns() - t0) > 50000000LL) return false;  // 50 ms
  }
  return true;
}

template <int NMAX, int RS, int SL, int ACCB, int DG, int NMW, int KS, bool BIN, bool FC1,
          bool CLAMP = false>
__global__ void __launch_bounds__(gemm_threads(DG), 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  using C = Cfg<NMAX, RS, SL, ACCB, DG, NMW, KS>;
  static_assert(BIN || KS == 1, "2-D pair-row boxes are issued per 128-wide block");
  // BIN: pair rows as one 3-D box {64, NMAX rows, 2 KS slabs} per step, copied by the
  // MMA warps; otherwise 2-D boxes of kPairBoxRows rows from a producer warp
  constexpr int kWeightTmaWarp = weight_tma_warp(BIN);
  constexpr int kPairTmaWarp = pair_tma_warp(BIN);
  // decode pipeline with tiles wider than 16 pairs: the warp after the MMA warps copies
  // the pair rows (3-D boxes), so that the MMA warps' per-step work is one wait and the
  // MMAs
  constexpr bool PB = BIN && NMAX > 16;
  constexpr int kPairBinWarp = kMmaWarp0 + NMW;
  static_assert(!PB || kPairBinWarp < kEpiWarp0, "a free warp for the pair-row copies");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bring = smem;                          // [SL][kBBytes] pair rows
  uint8_t* rring = smem + SL * C::kBBytes;        // [RS][kStageBytes]
  uint8_t* ctrl = rring + RS * C::kStageBytes;
  uint64_t* rfull = reinterpret_cast<uint64_t*>(ctrl);  // raw step landed (tx)
  uint64_t* rempty = rfull + RS;                        // raw step read by 4 dequant warps
  // sfull[slot * KS + h]: block h of the slot stored by the 4 dequant warps (block 0
  // also waits for the pair rows' bytes), so the MMAs of block 0 can start while the
  // dequant warps still work on block 1
  uint64_t* sfull = rempty + RS;
  uint64_t* sempty = sfull + SL * KS;                   // slot read by the MMAs
  uint64_t* accf = sempty + SL;                         // accumulators ready (NMW commits)
  uint64_t* acce = accf + ACCB;                         // accumulators drained (4 warps)
  uint64_t* drain = acce + ACCB;
  // 2-D pair-row boxes (no BIN): slab 0 of a slot may be refilled once the previous
  // step's slab-0 MMAs have completed (bempty0), slab 1 lands on its own barrier
  // (bfull1), so the copy of a slot's first slab starts half a step earlier
  uint64_t* bempty0 = drain + 1;
  uint64_t* bfull1 = bempty0 + SL;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfull1 + SL);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the E4M3 -> bf16x2 scale table at a fixed shared address, so that a lookup's
  // address is the byte's offset plus a constant (measured: decode layer 493 -> 480 µs
  // against the table in the dynamic area)
  __shared__ uint32_t scale_lut[256];
  uint8_t* epi_stage = ctrl + kCtrlBytes;  // [4][NMAX] ids, weights

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the route's tile count, read before the set-up below so that its latency overlaps it
  // (the route has completed before any GEMM of the forward starts)
  const int n_part_tiles = part_tiles(p);
  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(smem_u32(&rfull[s]), 1);
      mbar_init(smem_u32(&rempty[s]), 4);
    }
    for (int s = 0; s < SL; ++s) {
      // the pair rows' copy counts on block 0's barrier, or with the producer warp (PB)
      // on the last block's: there the MMA warp waits once per step, for every block
      for (int h = 0; h < KS; ++h)
        mbar_init(smem_u32(&sfull[s * KS + h]), h == (PB ? KS - 1 : 0) ? 5 : 4);
      mbar_init(smem_u32(&sempty[s]), 1);
    }
    for (int a = 0; a < ACCB; ++a) {
      mbar_init(smem_u32(&accf[a]), NMW);
      mbar_init(smem_u32(&acce[a]), 4);
    }
    mbar_init(smem_u32(drain), NMW);
    for (int s = 0; s < SL; ++s) {
      mbar_init(smem_u32(&bempty0[s]), 1);
      mbar_init(smem_u32(&bfull1[s]), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int b = threadIdx.x; b < 256; b += C::kThreads) scale_lut[b] = e4m3_scale_bf16x2(b);
  if (warp == kMmaWarp0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == (BIN ? kMmaWarp0 : kPairTmaWarp) && lane == 0) prefetch_tmap(&tmap_b);
  grid_dep_launch();  // the next kernel may take SMs as this grid's CTAs finish
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The CTA allocates all 512 TMEM columns, so the allocation can only start at lane 0,
  // column 0: the base is the constant 0, which lets the compiler keep the TMEM operands
  // of the MMAs uniform (measured with the MMA issue below: decode M=16 layer 479 -> 474
  // µs).  The address the allocation wrote is still checked.
  static_assert(kTmemCols == 512, "the constant TMEM base needs the whole TMEM");
  const uint32_t tmem = 0u;
  if (threadIdx.x == 0 && *tmem_slot != 0u && p.err) atomicOr(p.err, QMOE_FLAG_INTERNAL);

  const int nb128 = p.K / kBK;            // 128-wide weight blocks per unit
  const int nks = (nb128 + KS - 1) / KS;  // pipeline steps per unit
  const int last_halves = nb128 - (nks - 1) * KS;
  const int n_units = n_part_tiles * p.nrb;
  // BIN (decode, stream-K): the units' K steps form one sequence of n_units * nks steps,
  // cut into gridDim.x contiguous ranges, one per CTA; a unit split between CTAs is
  // summed from their partial accumulators in K order (sk_reduce).  Otherwise each CTA
  // takes whole units u = blockIdx.x, blockIdx.x + gridDim.x, ..
  const unsigned long long n_steps = (unsigned long long)n_units * (unsigned long long)nks;
  uint32_t g0 = 0, total = 0;
  if constexpr (BIN) {
    // units are split only with tiles of one 16-column chunk (the partial buffer's width)
    if (NMAX == 16 && sk_split(n_units, nks, gridDim.x)) {
      g0 = sk_range_start(n_steps, blockIdx.x, gridDim.x);
      total = sk_range_start(n_steps, blockIdx.x + 1, gridDim.x) - g0;
    } else {  // whole units: a contiguous run of them per CTA, no partial sums
      const uint32_t u0 = sk_range_start(n_units, blockIdx.x, gridDim.x);
      const uint32_t u1 = sk_range_start(n_units, blockIdx.x + 1, gridDim.x);
      g0 = u0 * (uint32_t)nks;
      total = (u1 - u0) * (uint32_t)nks;
    }
  } else {
    const int my_units =
        blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    total = (uint32_t)my_units * (uint32_t)nks;
  }

  if (warp == kWeightTmaWarp) {
    // ------------------------------------------------------------ weight TMA producer
    // (whole warp, converged; one elected lane issues)
    const uint32_t leader = elect_one();
    const uint64_t pol = l2_policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    // local step it: weights of step ks of unit u
    auto issue = [&](int u, int ks) -> bool {
      const int j = u / p.nrb, rb = u - j * p.nrb;
      const int e = p.tiles[3 * part_tile(p, j)];
      const size_t blk = ((size_t)e * p.nrb + rb) * (size_t)nb128;
      const int s = it % RS;
      if (!warp_wait(smem_u32(&rempty[s]), ((it / RS) & 1) ^ 1, abort_flag, p.err)) return false;
      const uint32_t nh = ks == nks - 1 ? (uint32_t)last_halves : (uint32_t)KS;
      const size_t b0 = blk + (size_t)ks * KS;
      const uint32_t st = smem_u32(rring + s * C::kStageBytes);
      const uint32_t fb = smem_u32(&rfull[s]);
      mbar_arrive_expect_tx_if(leader, fb, nh * kRawBytes);
      bulk_g2s_if(leader, st, p.wcodes + b0 * kCodeBytes, nh * kCodeBytes, fb, pol);
      bulk_g2s_if(leader, st + KS * kCodeBytes, p.wscales + b0 * kScaleBytes, nh * kScaleBytes,
                  fb, pol);
      return true;
    };
    if constexpr (BIN) {
      for (; it < total && ok; ++it) {
        const uint32_t g = g0 + it;
        const int u = (int)(g / (uint32_t)nks);
        ok = issue(u, (int)(g - (uint32_t)u * nks));
      }
    } else {
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x)
        for (int ks = 0; ks < nks && ok; ++ks, ++it) ok = issue(u, ks);
    }
    if (!ok) --it;  // the failed step was not issued
    if (!ok) {  // let the copies already issued land before the CTA can exit
      const uint32_t first = it > (uint32_t)RS ? it - RS : 0u;
      for (uint32_t j = first; j < it; ++j) drain_wait(smem_u32(&rfull[j % RS]), (j / RS) & 1);
    }
  } else if (!BIN && warp == kPairTmaWarp) {
    // ------------------------------------------------------------ pair-row TMA producer
    const uint32_t leader = elect_one();
    const uint64_t pol = l2_policy_evict_last();
    grid_dep_wait();  // the pair rows are the previous kernel's output
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int t = part_tile(p, u / p.nrb);
      const int start = p.tiles[3 * t + 1], rows = p.tiles[3 * t + 2];
      const int nbox = (rows + kPairBoxRows - 1) / kPairBoxRows;
      const uint32_t tx = (uint32_t)nbox * (uint32_t)(kPairBoxRows * 128);  // one slab
      for (int ks = 0; ks < nks && ok; ++ks, ++it) {
        const int s = it % SL;
        const uint32_t eph = ((it / SL) & 1) ^ 1;
        const uint32_t st = smem_u32(bring + s * C::kBBytes);
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
          // slab 0 is free once the slot's previous slab-0 MMAs completed, slab 1 once
          // the whole previous step did
          const uint32_t eb = smem_u32(sl == 0 ? &bempty0[s] : &sempty[s]);
          if (!warp_wait(eb, eph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(sl == 0 ? &sfull[s * KS] : &bfull1[s]);
          mbar_arrive_expect_tx_if(leader, fb, tx);
          for (int g = 0; g < nbox; ++g)
            tma_load_2d_if(leader, st + sl * C::kBSlab + g * kPairBoxRows * 128, &tmap_b,
                           ks * kBK + sl * 64, start + g * kPairBoxRows, fb, pol);
        }
      }
    }
    if (!ok) {  // the pair rows of the last slots may still be landing
      const unsigned long long t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
  } else if (PB && warp == kPairBinWarp) {
    // ------------------------------------------------------------ pair-row producer (PB)
    // step i's rows into slot i % SL once the MMAs of step i - SL completed
    const uint32_t leader = elect_one();
    const uint64_t bpol = l2_policy_evict_last();
    grid_dep_wait();  // the pair rows are the previous kernel's output
    bool ok = true;
    for (uint32_t bg = 0; bg < total && ok; ++bg) {
      const uint32_t g = g0 + bg;
      const int u = (int)(g / (uint32_t)nks);
      const int bks = (int)(g - (uint32_t)u * nks);
      const int bstart = p.tiles[3 * part_tile(p, u / p.nrb) + 1];
      const uint32_t sl = bg % SL;
      if (!warp_wait(smem_u32(&sempty[sl]), ((bg / SL) & 1) ^ 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&sfull[sl * KS + KS - 1]);
      mbar_arrive_expect_tx_if(leader, fb, (uint32_t)C::kBBytes);
      tma_load_3d_if(leader, smem_u32(bring + sl * C::kBBytes), &tmap_b, 0, bstart, 2 * KS * bks, fb,
                     bpol);
    }
    if (!ok) {  // the pair rows of the last slots may still be landing
      const unsigned long long t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + NMW) {
    // ------------------------------------------------------------ MMA issuers
    // MMA warp m takes the global K steps g with g % NMW == m, into its own accumulator.
    // Whole warp, converged; one elected lane issues.
    const int m = warp - kMmaWarp0;
    const uint32_t leader = elect_one();
    const uint32_t sfull_u = smem_u32(&sfull[0]), sempty_u = smem_u32(&sempty[0]);
    const uint32_t bempty0_u = smem_u32(&bempty0[0]), bfull1_u = smem_u32(&bfull1[0]);
    const uint64_t bdesc0 = sdesc_sw128(smem_u32(bring));
    const uint32_t bdesc_lo0 = (uint32_t)bdesc0, bdesc_hi = (uint32_t)(bdesc0 >> 32);
    uint32_t it = 0, local = 0;
    bool ok = true;
    // BIN: the pair rows of local step i go into slot i % SL, whose previous step
    // i - SL belongs to this warp too (SL % NMW == 0).  The copy for the warp's next
    // step is issued right after the MMAs of the current one, when the slot's previous
    // step (one own step back) has long completed: a step of lead for the copy.
    uint32_t bg = (uint32_t)m;  // local step of the next copy
    const uint64_t bpol = l2_policy_evict_last();
    auto issue_b = [&]() -> bool {
      if (bg >= total) return true;
      const uint32_t g = g0 + bg;
      const int u = (int)(g / (uint32_t)nks);
      const int bks = (int)(g - (uint32_t)u * nks);
      const int bstart = p.tiles[3 * part_tile(p, u / p.nrb) + 1];
      const uint32_t sl = bg % SL;
      if (!warp_wait(sempty_u + sl * 8, ((bg / SL) & 1) ^ 1, abort_flag, p.err)) return false;
      const uint32_t fb = sfull_u + sl * KS * 8;
      mbar_arrive_expect_tx_if(leader, fb, (uint32_t)C::kBBytes);
      tma_load_3d_if(leader, smem_u32(bring + sl * C::kBBytes), &tmap_b, 0, bstart,
                     2 * KS * bks, fb, bpol);
      bg += NMW;
      return true;
    };
    if constexpr (BIN && !PB) {
      grid_dep_wait();  // the pair rows are the previous kernel's output
      ok = issue_b();
    }
    // BIN: segments (the part of one unit inside this CTA's step range) one after the
    // other; otherwise whole units
    int u = BIN ? 0 : (int)blockIdx.x;
    while (ok && (BIN ? it < total : u < n_units)) {
      int k0 = 0, len = nks;
      if constexpr (BIN) {
        const uint32_t g = g0 + it;
        u = (int)(g / (uint32_t)nks);
        k0 = (int)(g - (uint32_t)u * nks);
        len = min(nks - k0, (int)(total - it));
      }
      const int t = part_tile(p, u / p.nrb);
      const int rows = p.tiles[3 * t + 2];
      const int n16 = ((rows + 15) >> 4) << 4;
      const uint32_t idesc = idesc_bf16_f32(128, n16 < 256 ? n16 : 256);
      // tiles wider than 256 pairs: a second chain over the rest (NMAX > 256 only)
      const uint32_t idesc2 = idesc_bf16_f32(128, n16 > 256 ? n16 - 256 : 16);
      const int ab = local % ACCB;
      if (!warp_wait(smem_u32(&acce[ab]), ((local / ACCB) & 1) ^ 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + C::kAccCol0 + (ab * NMW + m) * NMAX;
      // this warp's first step of the segment: local step it + ks with (it + ks) % NMW == m
      const int ks0 = (m - (int)(it % NMW) + NMW) % NMW;
      for (int ks = ks0; ks < len; ks += NMW) {
        const uint32_t sit = it + (uint32_t)ks;
        const int sl = sit % SL;
        const uint32_t sph = (sit / SL) & 1;
        // PB: the last block's barrier completes after every block of the step and its
        // pair rows; otherwise block 0's (the pair rows and block 0)
        if (!warp_wait(sfull_u + (sl * KS + (PB ? KS - 1 : 0)) * 8, sph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (!BIN) {
          // slab by slab: the first slab's stage is released (bempty0) as soon as its
          // MMAs complete, the second may still be landing (bfull1)
          const uint32_t a0 = tmem + sl * C::kSlotCols;
          const uint32_t b0 = bdesc_lo0 + sl * (C::kBBytes >> 4);
          const uint32_t acc = ks != ks0 ? 1u : 0u;
          // the MMAs are issued inside the elected lane's branch (see below)
          if (leader) {
            if (NMAX > 256 && n16 > 256)
              mma_bf16_ts_slab4x2(1u, d_tmem, d_tmem + 256, a0, b0, bdesc_hi, (256 * 128) >> 4,
                                  idesc, idesc2, acc);
            else
              mma_bf16_ts_slab4(1u, d_tmem, a0, b0, bdesc_hi, idesc, acc);
          }
          tc_commit_if(leader, bempty0_u + sl * 8);
          if (!warp_wait(bfull1_u + sl * 8, sph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b1 = b0 + (C::kBSlab >> 4);
          if (leader) {
            if (NMAX > 256 && n16 > 256)
              mma_bf16_ts_slab4x2(1u, d_tmem, d_tmem + 256, a0 + 32, b1, bdesc_hi,
                                  (256 * 128) >> 4, idesc, idesc2, 1u);
            else
              mma_bf16_ts_slab4(1u, d_tmem, a0 + 32, b1, bdesc_hi, idesc, 1u);
          }
        } else {
          // Issued inside the elected lane's branch rather than predicated per lane: with
          // operands the compiler can keep uniform the MMA warp's issue takes about half
          // the instructions (measured: decode FC2 -2.5%, skewed prefill FC1 -1%).
          if (leader)
            mma_bf16_ts_step8(1u, d_tmem, tmem + sl * C::kSlotCols,
                              bdesc_lo0 + sl * (C::kBBytes >> 4), bdesc_hi, C::kBSlab >> 4,
                              idesc, ks != ks0 ? 1u : 0u);
        }
        if (KS == 2 && (k0 + ks != nks - 1 || last_halves == 2)) {
          if (!PB && !warp_wait(sfull_u + (sl * KS + 1) * 8, sph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader)
            mma_bf16_ts_step8(1u, d_tmem, tmem + sl * C::kSlotCols + 64,
                              bdesc_lo0 + ((sl * C::kBBytes + 2 * C::kBSlab) >> 4), bdesc_hi,
                              C::kBSlab >> 4, idesc, 1u);
        }
        tc_commit_if(leader, sempty_u + sl * 8);
        if constexpr (BIN && !PB) {
          if (!issue_b()) {
            ok = false;
            break;
          }
        }
      }
      it += len;
      ++local;
      if constexpr (!BIN) u += gridDim.x;
      if (ok) tc_commit_if(leader, smem_u32(&accf[ab]));
    }
    // no MMA may still be running when TMEM is released
    tc_commit_if(leader, smem_u32(drain));
    drain_wait(smem_u32(drain), 0);
    if (BIN && !PB && !ok) {  // the pair rows of the last slots may still be landing
      const unsigned long long t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant warps (DG groups)
    const int grp = (warp - kDequantWarp0) >> 2;  // this group's steps: grp, grp + DG, ..
    const int q = warp & 3;                       // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;                // weight row of the 128-row block
    // The dequant warps only walk the CTA's step sequence.  RS and SL are multiples of
    // DG, so the group meets the same ring residues on every lap (s, a) and the phase
    // bits flip on each wrap.
    uint32_t s = grp, a = grp, rph = 0, aph = 0;
    uint32_t pos = (g0 + (uint32_t)grp) % (uint32_t)nks;  // step of the current one within its unit
    const DequantMul dqm{p.dq_mul[0], p.dq_mul[1]};
    for (uint32_t it = grp; it < total; it += DG) {
      const int nh = (KS == 2 && pos == (uint32_t)nks - 1) ? last_halves : KS;
      if (!warp_wait(smem_u32(&rfull[s]), rph, abort_flag, p.err)) break;
      const uint8_t* st = rring + s * C::kStageBytes;
      uint4 cw[KS][4];
      uint2 sc[KS];
#pragma unroll
      for (int h = 0; h < KS; ++h) {
        if (h < nh) {
          const uint4* codes = reinterpret_cast<const uint4*>(st + h * kCodeBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) cw[h][kk] = codes[kk * 128 + row];
          sc[h] = *reinterpret_cast<const uint2*>(st + KS * kCodeBytes + h * kScaleBytes + row * 8);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rempty[s]));  // the raw stage may be refilled
      if (!warp_wait(smem_u32(&sempty[a]), aph ^ 1, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + a * C::kSlotCols;
      // the row's block scales of every block of the step as bf16x2 multipliers, looked
      // up before the first TMEM store (whose ordering constraint would otherwise
      // serialize the lookups behind the stores)
      uint32_t sv[KS][8];
#pragma unroll
      for (int h = 0; h < KS; ++h) {
        if (h < nh) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            sv[h][j] = scale_lut[((j < 4 ? sc[h].x : sc[h].y) >> (8 * (j & 3))) & 0xFF];
        }
      }
#pragma unroll
      for (int h = 0; h < KS; ++h) {
        if (h < nh) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint32_t o[16];
            dequant8(cw[h][kk].x, sv[h][2 * kk], o + 0, dqm);
            dequant8(cw[h][kk].y, sv[h][2 * kk], o + 4, dqm);
            dequant8(cw[h][kk].z, sv[h][2 * kk + 1], o + 8, dqm);
            dequant8(cw[h][kk].w, sv[h][2 * kk + 1], o + 12, dqm);
            tmem_st_x16(ta + h * 64 + kk * 16, o);
          }
        }
        // PB: the MMA warp waits for the last block only, so one wait for the stores
        // serves all blocks; otherwise each block is published as soon as it is stored
        // (the MMAs of block 0 start while block 1 is converted)
        if (!PB || h == KS - 1) {
          if (PB || h < nh) {
            tmem_wait_st();
            tc_fence_before();
          }
          // a block past the unit's end is left unwritten, but its barrier still
          // completes so that every slot barrier advances once per use
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int b = PB ? 0 : h; b <= h; ++b) mbar_arrive(smem_u32(&sfull[a * KS + b]));
          }
        }
      }
      s += DG;
      if (s >= (uint32_t)RS) { s -= RS; rph ^= 1; }
      a += DG;
      if (a >= (uint32_t)SL) { a -= SL; aph ^= 1; }
      pos += DG;
      while (pos >= (uint32_t)nks) pos -= nks;
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;
    constexpr int NCH = NMAX / 16;          // 16-column chunks of a tile
    constexpr int G = NMW == 1 ? 4 : 1;     // chunks per TMEM round trip
    uint32_t local = 0, it0 = 0;
    int u = BIN ? 0 : (int)blockIdx.x;
    while (BIN ? it0 < total : u < n_units) {
      int k0 = 0, len = nks;
      if constexpr (BIN) {
        const uint32_t g = g0 + it0;
        u = (int)(g / (uint32_t)nks);
        k0 = (int)(g - (uint32_t)u * nks);
        len = min(nks - k0, (int)(total - it0));
      }
      const int j = u / p.nrb, rb = u - j * p.nrb;
      const int t = part_tile(p, j);
      const int e = p.tiles[3 * t], start = p.tiles[3 * t + 1], rows = p.tiles[3 * t + 2];
      const int ab = local % ACCB;
      const float gsc = p.gscale[e] * 128.0f;  // 2^7 undoes the dequant's 2^-7
      int* st_pair = reinterpret_cast<int*>(epi_stage + q * NMAX * 8);
      float* st_w = reinterpret_cast<float*>(st_pair + NMAX);
      if constexpr (!FC1 && !BIN) {
        epilogue_stage_fc2(p, lane, start, rows, gsc, st_pair, st_w);
        __syncwarp();
      }
      if (!warp_wait(smem_u32(&accf[ab]), (local / ACCB) & 1, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem + ((uint32_t)(q * 32) << 16) + C::kAccCol0 + ab * NMW * NMAX;
      if constexpr (BIN) {
        static_assert(!BIN || NMAX % 16 == 0, "16-column chunks");
        const bool whole = k0 == 0 && len == nks;  // always, unless NMAX == 16
        // the tile's 16-column chunks one after the other (decode: the only one)
        for (int c = 0; c < NMAX / 16; ++c) {
          if (c > 0 && 16 * c >= rows) break;
          float v[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = 0.f;
          // accumulators in the fixed order m = 0, 1, ..; warp m holds MMAs of this
          // segment iff its first step (m - it0 % NMW) mod NMW lies inside the segment
          for (int m = 0; m < NMW; ++m) {
            if ((m - (int)(it0 % NMW) + NMW) % NMW >= len) continue;
            uint32_t r[16];
            tmem_ld_x16(tbase + m * NMAX + 16 * c, r);
            tmem_wait_ld();
            tmem_ld_ready(r);
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] += __uint_as_float(r[k]);
          }
          if (c == NMAX / 16 - 1 || 16 * (c + 1) >= rows) {
            // the accumulator may be refilled once every warp has read it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce[ab]));
          }
          if (whole || (NMAX == 16 && sk_reduce(p, v, u, nks, n_steps, g0, lane, q)))
            epilogue_chunk_small<FC1, CLAMP>(p, v, lane, q, rb, start, rows, 16 * c, gsc);
        }
        it0 += len;
        ++local;
        continue;
      } else {
        // warp m holds MMAs of this unit iff its first step ks0 = (m - it0 % NMW) mod NMW
        // lies inside the unit; accumulators are added in the fixed order m = 0, 1, ..
        bool has[NMW];
#pragma unroll
        for (int m = 0; m < NMW; ++m) has[m] = (m - (int)(it0 % NMW) + NMW) % NMW < nks;
        // one batch body, reused (not unrolled: a smaller kernel, measurably faster)
#pragma unroll 1
        for (int kc = 0; kc < NCH; kc += G) {
          if (16 * kc >= rows) break;
          uint32_t r[NMW][G][16];
#pragma unroll
          for (int m = 0; m < NMW; ++m) {
            if (!has[m]) continue;
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (16 * (kc + g) < rows) tmem_ld_x16(tbase + m * NMAX + 16 * (kc + g), r[m][g]);
          }
          tmem_wait_ld();
#pragma unroll
          for (int m = 0; m < NMW; ++m) {
            if (!has[m]) continue;
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (16 * (kc + g) < rows) tmem_ld_ready(r[m][g]);
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int k = kc + g;
            if (16 * k >= rows) break;
            float v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = 0.f;
#pragma unroll
            for (int m = 0; m < NMW; ++m) {
              if (!has[m]) continue;
#pragma unroll
              for (int c = 0; c < 16; ++c) v[c] += __uint_as_float(r[m][g][c]);
            }
            if constexpr (FC1)
              epilogue_chunk_fc1_tr<CLAMP>(p, v, lane, q, rb, start, rows, 16 * k, gsc,
                                    reinterpret_cast<uint8_t*>(st_pair));
            else
              epilogue_chunk_fc2_staged(p, v, lane, q, rb, rows, 16 * k, st_pair, st_w);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acce[ab]));
      ++local;
      it0 += nks;
      u += gridDim.x;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NMAX, int RS, int SL, int ACCB, int DG, int NMW, int KS, bool BIN, bool FC1,
          bool CLAMP = false>
cudaError_t run(const CUtensorMap& tmap, const GemmParams& p, int num_sms, cudaStream_t stream,
               bool pdl = true) {
  using C = Cfg<NMAX, RS, SL, ACCB, DG, NMW, KS>;
  auto* k = moe_gemm_kernel<NMAX, RS, SL, ACCB, DG, NMW, KS, BIN, FC1, CLAMP>;
  cudaError_t rc = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (rc != cudaSuccess) return rc;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, tmap, p);
}

}  // namespace

bool forward_uses_pdl(int sched) { return sched != QMOE_SCHED_PREFILL; }

int gemm_tile_n(int sched) {
  if (sched == QMOE_SCHED_DECODE) return 16;
  if (sched == kSchedPrefillSmall) return kSmallTileRows;
  if (sched == QMOE_SCHED_PREFILL_PAIR) return 256;
  return sched == kSchedPrefillNarrow ? 192 : 320;
}

int gemm_b_box_rows(int sched) {
  if (sched == QMOE_SCHED_DECODE) return 16;
  return sched == kSchedPrefillSmall ? kSmallTileRows : kPairBoxRows;
}

int gemm_b_box_slabs(int sched) {
  return sched == QMOE_SCHED_DECODE || sched == kSchedPrefillSmall ? 4 : 0;
}

// decode : tiles <= 16 pairs, steps of 2 weight blocks (256 of K), 9 steps in flight
//          (162 KB), 3 slots, 3 MMA warps x 2 accumulator buffers, 3 dequant groups, pair
//          rows as one 3-D box per step
// prefill: one SM per tile: tiles <= 320 pairs (an expert of up to 320 routed pairs is
//          one tile, so its weights are dequantized once per row block), 6 weight
//          steps, 2 slots (80 KB of pair rows each), 1 MMA warp, 1 accumulator (320
//          columns: MMAs of N = 256 and of the rest), 2 dequant groups, 2-D boxes of
//          64 rows.  An MMA costs about the same for any N from about 160 to 256, so
//          wide tiles make the most of the tensor cores, at the price of an epilogue
//          that stalls the MMAs (one accumulator fills the TMEM);
//          narrow variant (experts averaging < 192 pairs): tiles <= 192 pairs, 8
//          weight steps, 2 accumulators, so the epilogue overlaps the next tile's MMAs
cudaError_t launch_gemm(GemmKind kind, int sched, const CUtensorMap& tmap_b, const GemmParams& p,
                        int num_sms, cudaStream_t stream) {
  const bool fc1 = kind == GemmKind::kFc1;
  // FC1 with a finite SwiGLU limit runs the clamping instantiations (the two-SM
  // schedule then runs as the one-SM prefill one)
  const bool clamp = fc1 && std::isfinite(p.swiglu_limit);
  if (sched == QMOE_SCHED_DECODE) {
    // stream-K: one CTA per SM, at most kMaxSkCtas (the partial buffer's slot pairs)
    const int g = num_sms < kMaxSkCtas ? num_sms : kMaxSkCtas;
    if (clamp) return run<16, 9, 3, 2, 3, 3, 2, true, true, true>(tmap_b, p, g, stream);
    return fc1 ? run<16, 9, 3, 2, 3, 3, 2, true, true>(tmap_b, p, g, stream)
               : run<16, 9, 3, 2, 3, 3, 2, true, false>(tmap_b, p, g, stream);
  }
  if (sched == kSchedPrefillSmall) {
    // the decode pipeline with tiles of up to 64 pairs: one MMA warp, three A slots
    // of 256 of K, 6 weight steps in flight, whole units per CTA
    const int g = num_sms < kMaxSkCtas ? num_sms : kMaxSkCtas;
    if (clamp) return run<64, 6, 3, 2, 3, 1, 2, true, true, true>(tmap_b, p, g, stream);
    return fc1 ? run<64, 6, 3, 2, 3, 1, 2, true, true>(tmap_b, p, g, stream)
               : run<64, 6, 3, 2, 3, 1, 2, true, false>(tmap_b, p, g, stream);
  }
  if (sched == QMOE_SCHED_PREFILL_PAIR && !clamp && p.nrb % 2 == 0 && num_sms >= 2)
    return launch_gemm2(kind, tmap_b, p, num_sms, stream);
  if (sched == kSchedPrefillNarrow) {
    if (clamp) return run<192, 8, 2, 2, 2, 1, 1, false, true, true>(tmap_b, p, num_sms, stream);
    return fc1 ? run<192, 8, 2, 2, 2, 1, 1, false, true>(tmap_b, p, num_sms, stream)
               : run<192, 8, 2, 2, 2, 1, 1, false, false>(tmap_b, p, num_sms, stream);
  }
  const bool pdl = forward_uses_pdl(sched);
  if (clamp) return run<320, 6, 2, 1, 2, 1, 1, false, true, true>(tmap_b, p, num_sms, stream, pdl);
  return fc1 ? run<320, 6, 2, 1, 2, 1, 1, false, true>(tmap_b, p, num_sms, stream, pdl)
             : run<320, 6, 2, 1, 2, 1, 1, false, false>(tmap_b, p, num_sms, stream, pdl);
}

}  // namespace qmoe
