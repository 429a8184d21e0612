// Two-SM grouped GEMM for the prefill schedule (tcgen05 cta_group::2).
//
// Same layer maths as the single-SM kernel (megamoe_rm.cu page, fc1_rm / fc2_rm), with
// a CTA pair (one cluster of 2 SMs) per unit:
//   unit = (tile of <= 256 pairs of one expert, pair of 128-row weight blocks);
//   CTA rank r dequantizes weight block 2p + r into its own TMEM (the MMA's A rows
//   128r .. 128r + 127) and loads half of the tile's pair rows (B columns
//   r N/2 .. r N/2 + N/2 - 1) into its own shared memory;
//   the rank-0 CTA issues one M = 256 MMA per 16-wide K slice that reads A from both
//   TMEMs and B from both shared memories and writes D rows 128r.. into CTA r's TMEM.
// Per SM, every pair row fetched from L2 and read by the tensor core serves 256 weight
// rows instead of 128: half the B traffic per FLOP of the single-SM M = 128 tile, which
// at N = 256 saturates the SM's shared-memory bandwidth.
//
// Synchronisation across the pair (all waits bounded, see common.cuh):
//   sfull[s]  (rank 0): 4 + 4 dequant warps (the peer's arrive remotely), rank 0's
//             pair-row producer (expecting both CTAs' bytes), and the bytes of both
//             halves (the peer's copies count on rank 0's barrier, cta_group::2);
//   sempty[s], accf[a], drain (both): one arrival each from rank 0's MMA commit,
//             multicast to both CTAs;
//   acce[a]   (rank 0): 4 + 4 epilogue warps.
// Parity waits cannot tell phase k from k+2; every slot and stage is filled and
// drained by single ordered streams (SL % DG == 0, RS % DG == 0), as in the
// single-SM kernel.
#include "common.cuh"
#include "dequant.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace qmoe {
namespace {

constexpr int kBK = 128;
constexpr int kCodeBytes = 8192;
constexpr int kScaleBytes = 1024;
constexpr int kRawBytes = kCodeBytes + kScaleBytes;
constexpr int kTmemCols = 512;
constexpr int kCtrlBytes = 1024;  // barriers, TMEM slot, abort flag
constexpr int kNmax = 256;             // pairs per tile (both CTAs)
constexpr int kHalfRows = kNmax / 2;   // pair rows per CTA
constexpr int kBoxRows = 64;           // rows of a 2-D pair-row box
constexpr int kBSlab = kHalfRows * 128;
constexpr int kBBytes = 2 * kBSlab;    // one 128-wide K step of this CTA's pair rows

// Warp roles (per CTA): 0 weight TMA, 1 MMA issue (rank 0) and TMEM allocation (both),
// 2 pair-row TMA, 3 idle, 4..7 epilogue, 8.. dequant.
constexpr int kWeightWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kPairWarp = 2;
constexpr int kEpiWarp0 = 4;
constexpr int kDequantWarp0 = 8;
__host__ __device__ constexpr int gemm2_threads(int groups) { return (kDequantWarp0 + 4 * groups) * 32; }

template <int RS, int SL, int DG>
struct Cfg2 {
  static constexpr int kAccCol0 = SL * 64;
  static constexpr int kSmemBytes = SL * kBBytes + RS * kRawBytes + 1024 + kCtrlBytes;
  static constexpr int kThreads = gemm2_threads(DG);
  static_assert(SL * 64 + kNmax <= kTmemCols, "TMEM budget");
  static_assert(SL % DG == 0 && RS % DG == 0, "each slot and stage needs one dequant group");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert((2 * RS + 2 * SL + 2 + 1) * 8 + 16 <= 1024, "barrier area");
};

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals may come from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* err) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((i & 3) == 0) {
      if (*abort_flag) return false;
      if ((long long)(globaltimer_ns() - t0) > kWaitLimitNs) {
        *abort_flag = 1;
        if (err) atomicOr(err, QMOE_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool warp_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* err) {
  return __all_sync(0xffffffffu, mbar_wait_cl(bar, parity, abort_flag, err));
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ---------------------------------------------------------------- tcgen05, CTA pair
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive once on the barrier at `bar` in both CTAs of the pair when the MMAs issued so
// far complete.
__device__ __forceinline__ void tc_commit2_both_if(uint32_t pred, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b16 m;\n\tsetp.ne.b32 p, %0, 0;\n\tmov.b16 m, 3;\n\t"
      "@p tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%1], m;\n\t}" ::"r"(pred),
      "r"(bar)
      : "memory");
}
// The 8 M = 256 MMAs of one 128-wide K step (layout as mma_bf16_ts_step8).
__device__ __forceinline__ void mma2_step8(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                           uint32_t desc_lo, uint32_t desc_hi, uint32_t slab16,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q, t;\n\t.reg .b64 d;\n\t.reg .b32 lo, a;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 q, %7, 0;\n\t"
      "setp.eq.u32 t, 0, 0;\n\t"
      "mov.b64 d, {%3, %4};\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [%2], d, %6, q;\n\t"
      "add.u32 lo, %3, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 8;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, %3, 4;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 16;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, %3, 6;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 24;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, %3, %5;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 32;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, lo, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 40;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, lo, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 48;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, lo, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 56;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::f16 [%1], [a], d, %6, t;\n\t}" ::"r"(pred),
      "r"(d_tmem), "r"(a_tmem), "r"(desc_lo), "r"(desc_hi), "r"(slab16), "r"(idesc),
      "r"(accumulate)
      : "memory");
}

// 2-D tensor copy into this CTA's shared memory whose completion is counted on a
// barrier given by its shared::cluster address, in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair_if(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                                    int x, int y, uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint "
      "[%1], [%2, {%3, %4}], [%5], %6;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

__device__ __forceinline__ bool drain_wait_cl(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait_cl(bar, parity)) {
    if ((long long)(globaltimer_ns() - t0) > 50000000LL) return false;  // 50 ms
  }
  return true;
}

template <int RS, int SL, int DG, bool FC1>
__global__ void __launch_bounds__(gemm2_threads(DG), 1)
    moe_gemm2_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  using C = Cfg2<RS, SL, DG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bring = smem;                          // [SL][kBBytes] this CTA's pair rows
  uint8_t* rring = smem + SL * kBBytes;           // [RS][kRawBytes]
  uint8_t* ctrl = rring + RS * kRawBytes;
  uint64_t* rfull = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* rempty = rfull + RS;
  uint64_t* sfull = rempty + RS;   // rank 0 only
  uint64_t* sempty = sfull + SL;
  uint64_t* accf = sempty + SL;
  uint64_t* acce = accf + 1;       // rank 0 only
  uint64_t* drain = acce + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ uint32_t scale_lut[256];  // at a fixed shared address (cheaper lookups)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(smem_u32(&rfull[s]), 1);
      mbar_init(smem_u32(&rempty[s]), 4);
    }
    for (int s = 0; s < SL; ++s) {
      mbar_init(smem_u32(&sfull[s]), 9);
      mbar_init(smem_u32(&sempty[s]), 1);
    }
    mbar_init(smem_u32(accf), 1);
    mbar_init(smem_u32(acce), 8);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int b = threadIdx.x; b < 256; b += C::kThreads) scale_lut[b] = e4m3_scale_bf16x2(b);
  if (warp == kMmaWarp) {
    tmem_alloc2(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish2();
  }
  if (warp == kPairWarp && lane == 0) prefetch_tmap(&tmap_b);
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int nks = p.K / kBK;
  const int half_units = p.nrb / 2;  // weight-block pairs per tile
  const int n_units = (*p.n_tiles) * half_units;
  const int cl = (int)cluster_index(), ncl = (int)cluster_count();
  const int my_units = cl < n_units ? (n_units - 1 - cl) / ncl + 1 : 0;
  const uint32_t total = (uint32_t)my_units * (uint32_t)nks;
  // rank 0's barriers as seen from this CTA
  const uint32_t sfull0 = peer_addr(smem_u32(&sfull[0]), 0);
  const uint32_t acce0 = peer_addr(smem_u32(acce), 0);

  if (warp == kWeightWarp) {
    // ------------------------------------------------------------ weight TMA producer
    const uint32_t lead = elect_one();
    const uint64_t pol = l2_policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    for (int u = cl; u < n_units && ok; u += ncl) {
      const int t = u / half_units, pp = u - t * half_units;
      const int rb = 2 * pp + (int)rank;
      const int e = p.tiles[3 * t];
      const size_t blk = ((size_t)e * p.nrb + rb) * (size_t)nks;
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const int s = it % RS;
        if (!warp_wait(smem_u32(&rempty[s]), ((it / RS) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t st = smem_u32(rring + s * kRawBytes);
        const uint32_t fb = smem_u32(&rfull[s]);
        mbar_arrive_expect_tx_if(lead, fb, kRawBytes);
        bulk_g2s_if(lead, st, p.wcodes + (blk + ks) * kCodeBytes, kCodeBytes, fb, pol);
        bulk_g2s_if(lead, st + kCodeBytes, p.wscales + (blk + ks) * kScaleBytes, kScaleBytes, fb,
                    pol);
      }
    }
    if (!ok) {
      const uint32_t first = it > (uint32_t)RS ? it - RS : 0u;
      for (uint32_t j = first; j < it; ++j) drain_wait_cl(smem_u32(&rfull[j % RS]), (j / RS) & 1);
    }
  } else if (warp == kPairWarp) {
    // ------------------------------------------------------------ pair-row TMA producer
    // this CTA's half of the tile's rows: columns rank*N/2 .. of the MMA's N
    const uint32_t lead = elect_one();
    const uint64_t pol = l2_policy_evict_last();
    grid_dep_wait();  // the pair rows are the previous kernel's output
    uint32_t it = 0;
    bool ok = true;
    for (int u = cl; u < n_units && ok; u += ncl) {
      const int t = u / half_units;
      const int start = p.tiles[3 * t + 1], rows = p.tiles[3 * t + 2];
      const int half = (((rows + 15) >> 4) << 4) / 2;
      const int row0 = start + (int)rank * half;
      const int nbox = (half + kBoxRows - 1) / kBoxRows;
      const uint32_t tx = 2u * (uint32_t)nbox * (uint32_t)(kBoxRows * 128);
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const int s = it % SL;
        if (!warp_wait_cl(smem_u32(&sempty[s]), ((it / SL) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t st = smem_u32(bring + s * kBBytes);
        // both halves complete on rank 0's slot barrier, which expects both
        if (leader) mbar_arrive_expect_tx_if(lead, smem_u32(&sfull[s]), 2 * tx);
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
          for (int g = 0; g < nbox; ++g)
            tma_load_2d_pair_if(lead, st + sl * kBSlab + g * kBoxRows * 128, &tmap_b,
                                ks * kBK + sl * 64, row0 + g * kBoxRows, sfull0 + s * 8, pol);
      }
    }
    if (!ok) {  // the pair rows of the last slots may still be landing
      const unsigned long long t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
  } else if (warp == kMmaWarp && leader) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    const uint32_t lead = elect_one();
    const uint32_t sfull_u = smem_u32(&sfull[0]), sempty_u = smem_u32(&sempty[0]);
    const uint64_t bdesc0 = sdesc_sw128(smem_u32(bring));
    const uint32_t bdesc_lo0 = (uint32_t)bdesc0, bdesc_hi = (uint32_t)(bdesc0 >> 32);
    uint32_t it = 0, local = 0;
    bool ok = true;
    for (int u = cl; u < n_units && ok; u += ncl, ++local) {
      const int t = u / half_units;
      const int rows = p.tiles[3 * t + 2];
      const uint32_t idesc = idesc_bf16_f32(256, ((rows + 15) >> 4) << 4);
      if (!warp_wait_cl(smem_u32(acce), (local & 1) ^ 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + C::kAccCol0;
      for (int ks = 0; ks < nks; ++ks, ++it) {
        const int sl = it % SL;
        if (!warp_wait_cl(sfull_u + sl * 8, (it / SL) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // issued inside the elected lane's branch, as in the single-SM kernel
        if (lead)
          mma2_step8(1u, d_tmem, tmem + sl * 64, bdesc_lo0 + sl * (kBBytes >> 4), bdesc_hi,
                     kBSlab >> 4, idesc, ks != 0 ? 1u : 0u);
        tc_commit2_both_if(lead, sempty_u + sl * 8);
      }
      if (ok) tc_commit2_both_if(lead, smem_u32(accf));
    }
    tc_commit2_both_if(lead, smem_u32(drain));
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant warps
    const int grp = (warp - kDequantWarp0) >> 2;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const DequantMul dqm{p.dq_mul[0], p.dq_mul[1]};
    uint32_t s = grp, a = grp, rph = 0, aph = 0;
    for (uint32_t it = grp; it < total; it += DG) {
      if (!warp_wait(smem_u32(&rfull[s]), rph, abort_flag, p.err)) break;
      const uint8_t* st = rring + s * kRawBytes;
      const uint4* codes = reinterpret_cast<const uint4*>(st);
      uint4 cw[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) cw[kk] = codes[kk * 128 + row];
      const uint2 sc = *reinterpret_cast<const uint2*>(st + kCodeBytes + row * 8);
      uint32_t sv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) sv[j] = scale_lut[((j < 4 ? sc.x : sc.y) >> (8 * (j & 3))) & 0xFF];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rempty[s]));
      if (!warp_wait_cl(smem_u32(&sempty[a]), aph ^ 1, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + a * 64;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t o[16];
        dequant8(cw[kk].x, sv[2 * kk], o + 0, dqm);
        dequant8(cw[kk].y, sv[2 * kk], o + 4, dqm);
        dequant8(cw[kk].z, sv[2 * kk + 1], o + 8, dqm);
        dequant8(cw[kk].w, sv[2 * kk + 1], o + 12, dqm);
        tmem_st_x16(ta + kk * 16, o);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(smem_u32(&sfull[a]));
        else
          mbar_arrive_remote(sfull0 + a * 8);
      }
      s += DG;
      if (s >= (uint32_t)RS) { s -= RS; rph ^= 1; }
      a += DG;
      if (a >= (uint32_t)SL) { a -= SL; aph ^= 1; }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;
    uint32_t local = 0;
    for (int u = cl; u < n_units; u += ncl, ++local) {
      const int t = u / half_units, pp = u - t * half_units;
      const int rb = 2 * pp + (int)rank;
      const int e = p.tiles[3 * t], start = p.tiles[3 * t + 1], rows = p.tiles[3 * t + 2];
      const float gsc = p.gscale[e] * 128.0f;
      if (!warp_wait_cl(smem_u32(accf), local & 1, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + C::kAccCol0;
      // four chunks of 16 columns per TMEM round trip
#pragma unroll
      for (int k0 = 0; k0 < kNmax / 16; k0 += 4) {
        if (16 * k0 >= rows) break;
        uint32_t r[4][16];
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (16 * (k0 + g) < rows) tmem_ld_x16(tbase + 16 * (k0 + g), r[g]);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (16 * (k0 + g) < rows) tmem_ld_ready(r[g]);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int k = k0 + g;
          if (16 * k >= rows) break;
          float v[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(r[g][c]);
          if constexpr (FC1)
            epilogue_chunk_fc1(p, v, lane, q, rb, start, rows, 16 * k, gsc);
          else
            epilogue_chunk_small<false>(p, v, lane, q, rb, start, rows, 16 * k, gsc);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(smem_u32(acce));
        else
          mbar_arrive_remote(acce0);
      }
    }
  }

  // No MMA may still read this CTA's TMEM or shared memory, and no remote arrival may
  // still be in flight, when either CTA of the pair releases TMEM or exits.
  if (warp == kMmaWarp) drain_wait_cl(smem_u32(drain), 0);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc2(tmem, kTmemCols);
  }
}

template <int RS, int SL, int DG, bool FC1>
cudaError_t run2(const CUtensorMap& tmap, const GemmParams& p, int num_sms, cudaStream_t stream) {
  using C = Cfg2<RS, SL, DG>;
  auto* k = moe_gemm2_kernel<RS, SL, DG, FC1>;
  cudaError_t rc = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (rc != cudaSuccess) return rc;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // one CTA pair per pair of SMs that can hold it
  cfg.gridDim = dim3((unsigned)(num_sms & ~1));
  int clusters = 0;
  rc = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg);
  if (rc != cudaSuccess) return rc;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  if (2 * clusters < (int)cfg.gridDim.x) cfg.gridDim = dim3((unsigned)(2 * clusters));
  return cudaLaunchKernelEx(&cfg, k, tmap, p);
}

}  // namespace

// prefill, CTA pairs: tiles <= 256 pairs, 8 weight steps, 4 slots (32 KB of pair rows
// each per CTA), 1 accumulator (256 columns), 2 dequant groups
cudaError_t launch_gemm2(GemmKind kind, const CUtensorMap& tmap_b, const GemmParams& p, int num_sms,
                         cudaStream_t stream) {
  return kind == GemmKind::kFc1 ? run2<8, 4, 2, true>(tmap_b, p, num_sms, stream)
                                : run2<8, 4, 2, false>(tmap_b, p, num_sms, stream);
}

}  // namespace qmoe
