// dK/dV kernel of the deterministic backward on CTA pairs: the four products
// per (key block, query block) as 2-CTA tensor-core MMAs (tcgen05, cta_group::2).
//
// "Interrogating the GPU part 5: FlashAttention", "What does the backward pass
// do without P?" (recompute P from Q, K and the LSE; dV = P^T dO; dS =
// P o (dP - delta)) and "Why did Blackwell need FlashAttention-4?" (the 2-SM
// MMA: two SMs compute one 256-row product, each reading half of the other
// operand from its own shared memory).
//
// The work is the same as fa_bwd_kernel<D, CAUSAL, false> (dK and dV; dQ is
// left to the query-major pass): per key block j and each of its query
// blocks i, in the transposed orientation (TMEM lane = key),
//   S^T = K_j Q_i^T, dP^T = V_j dO_i^T          (issuer A)
//   P^T = 2^(S^T c - L_i log2e), dS^T = P^T o (dP^T - delta_i)
//                                               (elementwise warps, thread = key)
//   dV += P^T dO_i, dK += dS^T Q_i              (issuer B)
// A cluster of two CTAs takes the key blocks 2jp (rank 0, the leader) and
// 2jp + 1 (rank 1) of one (batch, head), and both walk the same query blocks
// in step: with the mask, from i = 2jp, where every key of rank 1's block is
// in the future, so its probabilities are 0 there.  (A last key block without
// a partner, for an odd number of blocks, is paired with a block past N: its
// keys read as zero and its dK, dV rows are not stored.)
//
// Every product is one 256-row MMA issued by the leader: rows 0-127 are the
// leader's keys, 128-255 the peer's, each in its own shared memory (K_j, V_j,
// dS^T) or tensor memory (P^T); the other operand's N columns are split in
// halves between the two CTAs.  So each CTA holds, per query block,
//   a row half of Q_i and of dO_i: queries [64 rank, 64 rank + 64), all d
//     columns (the B of S^T and dP^T, N = queries), and
//   a column half: all 128 queries, d columns [64 rank, 64 rank + 64) (the B
//     of dK and dV, N = d),
// 32 KB per tile, as much as a whole tile, but the tensor cores of the two SMs
// each read only half of every B operand.  Each CTA's TMA loads complete on
// the leader's barriers (kv_full, ring_full), the leader's commits arrive on
// both CTAs' barriers (multicast), and the peer's elementwise warps report
// P^T and dS^T written with one remote arrival per warp on the leader's
// p_done / ew_done.  The elementwise step, the statistics and the dK, dV
// write-out are each CTA's own, as in fa_bwd_kernel.
//
// Warp roles (512 threads): warps 0-7 elementwise; warp 12 issuer A and TMEM
// owner (the peer's only allocates); warp 13 TMA producer; warp 14 issuer B
// (leader only); warps 8-11 and 15 idle.  d = 128 only (at d = 64 a column half
// would be half a 128-byte swizzle atom).
#pragma once

#include <cuda_bf16.h>

#include <math_constants.h>

#include "sm103_ptx.cuh"
#include "fa_bwd.cuh"

namespace fa {

struct BwdPairCfg {
  static constexpr int D = 128;
  static constexpr int kTileBytes = 128 * D * 2;   // K_j, V_j, dS^T; and a ring slot (two halves)
  static constexpr int kHalfBytes = kTileBytes / 2;
  static constexpr int kRowHalfAtomBytes = 64 * 128;  // 64 rows x 64 columns: one atom column of a row half
  static constexpr int kSlots = 4;                 // Q / dO ring: Q_i at fill 2g, dO_i at 2g + 1
  static constexpr int kStatBytes = 1024;
  static constexpr int kStatEntries = kSlots / 2;  // statistics of the query blocks in flight (as fa_bwd_kernel)
  static constexpr int kDsBytes = 128 * 128 * 2;
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kDkCol = 0, kDvCol = D, kSCol = 2 * D, kDpCol = 2 * D + 128;
  static constexpr int kBarrierBytes = 512;
  static constexpr int kSmemBytes =
      2 * kTileBytes + kSlots * kTileBytes + kDsBytes + kStatEntries * kStatBytes + kBarrierBytes;
};

// Register budgets after setmaxnreg (the block launches with 128 per thread):
// the idle warpgroup (warps 8-11) gives most of its share to the elementwise
// warpgroups and the issuing/producer one: 2 x 168 + 56 + 96 = 488 <= 4 x 128.
constexpr uint32_t kPairWorkRegs = 168, kPairIdleRegs = 56, kPairMiscRegs = 96;
static_assert(2 * kPairWorkRegs + kPairIdleRegs + kPairMiscRegs <= 4 * 128, "register split above the launch budget");

struct BwdPairBarriers {
  uint64_t kv_full;        // (leader) K_j, V_j of both CTAs have landed
  uint64_t ring_full[4];   // (leader) both CTAs' halves of the fill have landed
  uint64_t ring_empty[4];  // (both, multicast) the fill's tile has been read by its last product
  uint64_t stat_full[2];   // (own) the statistics of a query block have landed
  uint64_t s_full, dp_full, dv_done, dk_done, acc_done;  // (both, multicast commits)
  uint64_t p_done, ew_done;  // (leader) the elementwise steps of both CTAs are written
  uint64_t drain[2];
  uint64_t never;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdPairBarriers) <= BwdPairCfg::kBarrierBytes, "barriers overflow their shared-memory slot");

enum : int { kSitePairProducer = 48, kSitePairKV, kSitePairQ, kSitePairDo, kSitePairDvDone, kSitePairEwPrev,
             kSitePairP, kSitePairEw, kSitePairS, kSitePairDp, kSitePairDk, kSitePairAcc, kSitePairStat };

// Items: pairs of key blocks (2jp, 2jp + 1) of one (batch, head), in the orders
// of bwd_item (without the mask head-major; with it grouped by heads,
// costliest first) with jp in place of the key block.
struct BwdPairItem {
  int bh, jb, i_start, n_it;
};
template <bool CAUSAL>
__device__ __forceinline__ BwdPairItem bwd_pair_item(const BwdParams& p, int k, int rank) {
  const int nj = (p.nkb + 1) >> 1;
  BwdPairItem t;
  int jp;
  if (CAUSAL) {
    const int per_group = p.group_heads * nj;
    const int grp = k / per_group;
    const int r = k - grp * per_group;
    const int gh = min(p.group_heads, p.num_bh - grp * p.group_heads);
    jp = r / gh;
    t.bh = grp * p.group_heads + (r - jp * gh);
  } else {
    t.bh = k / nj;
    jp = k - t.bh * nj;
  }
  t.jb = 2 * jp + rank;
  t.i_start = CAUSAL ? 2 * jp : 0;
  t.n_it = p.nkb - t.i_start;
  return t;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(512, 1)
    fa_bwd_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                       const __grid_constant__ CUtensorMap map_lse2, const __grid_constant__ CUtensorMap map_delta,
                       const __grid_constant__ CUtensorMap map_q64, const __grid_constant__ CUtensorMap map_do64,
                       const BwdParams p) {
  using C = BwdPairCfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // (both CTAs of a pair see the same alignment, so both return here or neither does)
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(&g_fa_device_status, 0u, kStatusBadSmem);
    return;
  }
  uint8_t* sK = smem_raw;
  uint8_t* sV = sK + C::kTileBytes;
  uint8_t* sRing = sV + C::kTileBytes;  // slot s: row half at +0 (two 8 KB atom columns), column half at +16 KB
  uint8_t* sDS = sRing + C::kSlots * C::kTileBytes;
  uint8_t* sStat = sDS + C::kDsBytes;
  BwdPairBarriers* bar = reinterpret_cast<BwdPairBarriers*>(sStat + C::kStatEntries * C::kStatBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  const int rank = (int)cluster_ctarank();
  const bool leader = rank == 0;

  if (tid == 0) {
    mbar_init(&bar->kv_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar->ring_full[s], 1);
      mbar_init(&bar->ring_empty[s], 1);
    }
    for (int e = 0; e < C::kStatEntries; ++e) mbar_init(&bar->stat_full[e], 1);
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->dp_full, 1);
    mbar_init(&bar->dv_done, 1);
    mbar_init(&bar->dk_done, 1);
    mbar_init(&bar->acc_done, 1);
    // the leader's 256 elementwise threads, and one arrival per peer elementwise warp
    mbar_init(&bar->p_done, 256 + 8);
    mbar_init(&bar->ew_done, 256 + 8);
    mbar_init(&bar->drain[0], 1);
    mbar_init(&bar->drain[1], 1);
    mbar_init(&bar->never, 1);
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc_pair(&bar->tmem_base, C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_k);
    tma_prefetch_map(&map_v);
    tma_prefetch_map(&map_do);
    tma_prefetch_map(&map_lse2);
    tma_prefetch_map(&map_delta);
    tma_prefetch_map(&map_q64);
    tma_prefetch_map(&map_do64);
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before either reaches into the other
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtx ctx{&bar->abort_flag, p.wait_limit_ns};
  // the leader's barriers that the peer's loads and elementwise warps complete
  const uint32_t lead_kv_full = mapa_shared(smem_u32(&bar->kv_full), 0);
  const uint32_t lead_p_done = mapa_shared(smem_u32(&bar->p_done), 0);
  const uint32_t lead_ew_done = mapa_shared(smem_u32(&bar->ew_done), 0);
  const int first = (int)(blockIdx.x >> 1), stride = (int)(gridDim.x >> 1);

  if (warp >= 12) {
    setmaxnreg_dec<kPairMiscRegs>();
    if (warp == 13) {
      // ------------------------------------------------------------------ TMA producer (both CTAs)
      if (lane == 0) {
        int fill = 0, g = 0, w = 0;
        bool ok = true;
        for (int item = first; ok && item < p.num_items; item += stride, ++w) {
          const BwdPairItem t = bwd_pair_item<CAUSAL>(p, item, rank);
          // K_j, V_j, once the previous item's last products have read the old ones
          if (w > 0 && !(ok = wait_bounded_cluster_inl(&bar->acc_done, (w - 1) & 1, ctx, kSitePairProducer))) break;
          if (leader) mbar_arrive_expect_tx(&bar->kv_full, 2 * 2 * C::kTileBytes);
          for (int a = 0; a < 2; ++a) {
            tma_load_3d_pair(sK + a * 16384, &map_k, lead_kv_full, a * 64, t.jb * 128, t.bh);
            tma_load_3d_pair(sV + a * 16384, &map_v, lead_kv_full, a * 64, t.jb * 128, t.bh);
          }
          for (int it = 0; ok && it < t.n_it; ++it, ++g) {
            const int i = t.i_start + it;
            for (int which = 0; which < 2; ++which) {
              const int s = fill % C::kSlots;
              const uint32_t u = fill / C::kSlots;
              if (!(ok = wait_bounded_cluster_inl(&bar->ring_empty[s], (u & 1) ^ 1, ctx, kSitePairProducer))) break;
              if (leader) mbar_arrive_expect_tx(&bar->ring_full[s], 2 * C::kTileBytes);
              const uint32_t lead_full = mapa_shared(smem_u32(&bar->ring_full[s]), 0);
              uint8_t* slot = sRing + s * C::kTileBytes;
              const CUtensorMap* m64 = which ? &map_do64 : &map_q64;
              const CUtensorMap* m128 = which ? &map_do : &map_q;
              // row half: queries [64 rank, 64 rank + 64) of block i, both atom columns
              for (int a = 0; a < 2; ++a)
                tma_load_3d_pair(slot + a * C::kRowHalfAtomBytes, m64, lead_full, a * 64, i * 128 + 64 * rank, t.bh);
              // column half: all 128 queries, atom column `rank`
              tma_load_3d_pair(slot + C::kHalfBytes, m128, lead_full, 64 * rank, i * 128, t.bh);
              if (!which) {
                // this CTA's statistics of block i (its own barrier); the entry was last
                // read by block g - kStatEntries, whose products have freed this slot
                const int e = g % C::kStatEntries;
                uint8_t* st = sStat + e * C::kStatBytes;
                mbar_arrive_expect_tx(&bar->stat_full[e], C::kStatBytes);
                tma_load_2d(st, &map_lse2, &bar->stat_full[e], i * 128, t.bh);
                tma_load_2d(st + 512, &map_delta, &bar->stat_full[e], i * 128, t.bh);
              }
              ++fill;
            }
          }
        }
        // the statistics loads must land before the CTA ends (the tile loads are
        // counted on the leader's barriers, which the leader's issuers wait for)
        // (entry e was loaded for the blocks b < g with b % kStatEntries == e;
        // only a Q fill that went out loads statistics, so count those: g
        // blocks finished their Q fill, plus one if the loop stopped after it)
        const int q_fills = (fill + 1) / 2;
        for (int e = 0; e < C::kStatEntries; ++e) {
          const int loads = (q_fills + C::kStatEntries - 1 - e) / C::kStatEntries;
          if (loads > 0) wait_drain_inl(&bar->stat_full[e], (loads - 1) & 1, kDrainLimitNs);
        }
        if (leader) {
          if (w > 0) wait_drain_cluster_inl(&bar->kv_full, (w - 1) & 1, kDrainLimitNs);
          for (int s = 0; s < C::kSlots; ++s)
            if (fill > s) {
              const int uses = (fill - 1 - s) / C::kSlots + 1;
              wait_drain_cluster_inl(&bar->ring_full[s], (uses - 1) & 1, kDrainLimitNs);
            }
        }
      }
      __syncwarp();
    } else if (warp == 12 && leader) {
      // ------------------------------------------------------------------ issuer A (leader): S^T and dP^T
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16_f32(256, 128, false, false);
        const uint32_t ring = smem_u32(sRing);
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint32_t tS = tmem + C::kSCol, tDP = tmem + C::kDpCol;
        bool ok = !(p.debug_stall && !wait_bounded_inl(&bar->never, 0, ctx, kSiteStall));
        int g = 0, w = 0;
        for (int item = first; ok && item < p.num_items; item += stride, ++w) {
          const BwdPairItem t = bwd_pair_item<CAUSAL>(p, item, rank);
          ok = wait_bounded_cluster_inl(&bar->kv_full, w & 1, ctx, kSitePairKV);
          for (int it = 0; ok && it < t.n_it; ++it, ++g) {
#pragma unroll
            for (int step = 0; step < 2; ++step) {
              const int f = 2 * g + step, s = f % C::kSlots;
              if (!(ok = wait_bounded_cluster_inl(&bar->ring_full[s], (f / C::kSlots) & 1, ctx,
                                                  step ? kSitePairDo : kSitePairQ)))
                break;
              // S^T overwrites the previous P^T (read by dV), dP^T the previous
              // dP^T (read by both CTAs' elementwise step)
              if (g > 0 && !(ok = step ? wait_bounded_cluster_inl(&bar->ew_done, (g - 1) & 1, ctx, kSitePairEwPrev)
                                       : wait_bounded_cluster_inl(&bar->dv_done, (g - 1) & 1, ctx, kSitePairDvDone)))
                break;
              tc_fence_after();
              const uint64_t bdesc = sdesc_sw128(ring + s * C::kTileBytes, 16, 1024);  // row half, K-major
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off_a = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                const uint32_t off_b = (uint32_t)(((kk >> 2) * C::kRowHalfAtomBytes + (kk & 3) * 32) >> 4);
                mma_bf16_ss_pair(step ? tDP : tS, (step ? vdesc : kdesc) + off_a, bdesc + off_b, id_s,
                                 kk > 0 ? 1u : 0u);
              }
              mma_commit_pair(step ? &bar->dp_full : &bar->s_full);
            }
          }
        }
        mma_commit_pair(&bar->drain[0]);
        wait_drain_cluster_inl(&bar->drain[0], 0, kDrainLimitNs);
      }
      __syncwarp();
    } else if (warp == 14 && leader) {
      // ------------------------------------------------------------------ issuer B (leader): dV and dK
      if (lane == 0) {
        constexpr uint32_t id_v = idesc_bf16_f32(256, D, false, true);
        const uint32_t ring = smem_u32(sRing);
        const uint64_t dsdesc_k = sdesc_sw128(smem_u32(sDS), 16, 1024);
        const uint32_t tS = tmem + C::kSCol;
        const uint32_t tDK = tmem + C::kDkCol, tDV = tmem + C::kDvCol;
        bool ok = true;
        int g = 0;
        for (int item = first; ok && item < p.num_items; item += stride) {
          const BwdPairItem t = bwd_pair_item<CAUSAL>(p, item, rank);
          for (int it = 0; ok && it < t.n_it; ++it, ++g) {
            const int sq = (2 * g) % C::kSlots, sd = (2 * g + 1) % C::kSlots;
            // dV += P^T dO_i once both CTAs' P^T is written (and dP^T, which also
            // read dO_i's row half, is complete): P^T of query group kk at S^T column 16 kk
            ok = wait_bounded_cluster_inl(&bar->dp_full, g & 1, ctx, kSitePairP) &&
                 wait_bounded_cluster_inl(&bar->p_done, g & 1, ctx, kSitePairP);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dodesc_mn = sdesc_sw128(ring + sd * C::kTileBytes + C::kHalfBytes, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ts_pair(tDV, tS + kk * 16, dodesc_mn + (uint32_t)((kk * 2048) >> 4), id_v,
                               (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit_pair(&bar->dv_done);
            mma_commit_pair(&bar->ring_empty[sd]);
            // dK += dS^T Q_i once both CTAs' dS^T is written
            if (!(ok = wait_bounded_cluster_inl(&bar->ew_done, g & 1, ctx, kSitePairEw))) break;
            tc_fence_after();
            const uint64_t qdesc_mn = sdesc_sw128(ring + sq * C::kTileBytes + C::kHalfBytes, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
              mma_bf16_ss_pair(tDK, dsdesc_k + off, qdesc_mn + (uint32_t)((kk * 2048) >> 4), id_v,
                               (it > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_pair(&bar->ring_empty[sq]);
            mma_commit_pair(&bar->dk_done);
          }
          if (ok) mma_commit_pair(&bar->acc_done);
        }
        mma_commit_pair(&bar->drain[1]);
        wait_drain_cluster_inl(&bar->drain[1], 0, kDrainLimitNs);
      }
      __syncwarp();
    }
    // warp 15, and the peer's issuing warps, have no role
  } else if (warp >= 8) {
    // warps 8-11: no role
    setmaxnreg_dec<kPairIdleRegs>();
  } else {
    // ------------------------------------------------------------------ elementwise (both CTAs)
    setmaxnreg_inc<kPairWorkRegs>();
    const int grp = warp >> 2;  // query columns [64 grp, 64 grp + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + C::kSCol + lane_off;
    const uint32_t tDP = tmem + C::kDpCol + lane_off;
    const float sl2 = p.scale_log2;
    uint8_t* ds_row = sDS + grp * 16384 + r * 128;
    bool alive = true;
    int g = 0, w = 0;
    // When this warp's part of an elementwise step is written, the leader's
    // threads arrive on its barrier one by one, the peer's warps once each, remotely.
#define FA_PAIR_REPORT(own_bar, lead_bar)        \
  do {                                           \
    if (leader) {                                \
      mbar_arrive(own_bar);                      \
    } else {                                     \
      __syncwarp();                              \
      if (lane == 0) mbar_arrive_remote(lead_bar); \
    }                                            \
  } while (0)
    for (int item = first; alive && item < p.num_items; item += stride, ++w) {
      const BwdPairItem t = bwd_pair_item<CAUSAL>(p, item, rank);
      for (int it = 0; alive && it < t.n_it; ++it, ++g) {
        const int i = t.i_start + it;
        const int e = g % C::kStatEntries;
        const float* stat = reinterpret_cast<const float*>(sStat + e * C::kStatBytes);
        // ---- phase 1: P^T = 2^(S^T c - L log2e) into TMEM, the fp32 values kept
        if (!__all_sync(0xffffffffu, wait_bounded_cluster_inl(&bar->s_full, g & 1, ctx, kSitePairS) &&
                                         wait_bounded_inl(&bar->stat_full[e], (g / C::kStatEntries) & 1, ctx,
                                                          kSitePairStat))) {
          alive = false;
          break;
        }
        tc_fence_after();
        // with the mask: key jb*128 + r is in the future of query i*128 + q when
        // q + (i - jb)*128 < r (i = jb: the diagonal; i < jb: every query)
        const bool masked_block = CAUSAL && i <= t.jb;
        const int qshift = (i - t.jb) * 128;
        const float2 c2 = make_float2(sl2, sl2);
        float2 pf[2][16];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int qc = 64 * grp + 32 * ch;
          uint32_t sv[32];
          tmem_ld32(tS + qc, sv);
          tmem_wait_ld();
          reg_fence32(sv);
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 l4 = *reinterpret_cast<const float4*>(stat + qc + 4 * e4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e2 = 4 * e4 + 2 * h;
              const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
              const float2 xs = __ffma2_rn(make_float2(__uint_as_float(sv[e2]), __uint_as_float(sv[e2 + 1])), c2, nl);
              float2 pe = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
              if (masked_block) {
                if (qc + e2 + qshift < r) pe.x = 0.f;
                if (qc + e2 + 1 + qshift < r) pe.y = 0.f;
              }
              pf[ch][e2 / 2] = pe;
              pk[2 * e4 + h] = pack_bf16x2(pe.x, pe.y);
            }
          }
          tmem_st8(tS + qc, pk);
          tmem_st8(tS + qc + 16, pk + 8);
        }
        tmem_wait_st();
        tc_fence_before();
        FA_PAIR_REPORT(&bar->p_done, lead_p_done);

        // ---- phase 2: dS^T = P^T o (dP^T - delta) into the shared dS^T tile, once
        // the previous block's dK has read it
        bool ok2 = wait_bounded_cluster_inl(&bar->dp_full, g & 1, ctx, kSitePairDp);
        if (g > 0) ok2 = ok2 && wait_bounded_cluster_inl(&bar->dk_done, (g - 1) & 1, ctx, kSitePairDk);
        if (!__all_sync(0xffffffffu, ok2)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int qc = 64 * grp + 32 * ch;
          uint32_t dp[32];
          tmem_ld32(tDP + qc, dp);
          tmem_wait_ld();
          reg_fence32(dp);
          uint32_t dk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 d4 = *reinterpret_cast<const float4*>(stat + 128 + qc + 4 * e4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e2 = 4 * e4 + 2 * h;
              const float2 nd = h ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
              const float2 dpd = __fadd2_rn(make_float2(__uint_as_float(dp[e2]), __uint_as_float(dp[e2 + 1])), nd);
              const float2 dse = __fmul2_rn(pf[ch][e2 / 2], dpd);
              dk[2 * e4 + h] = pack_bf16x2(dse.x, dse.y);
            }
          }
#pragma unroll
          for (int c16 = 0; c16 < 4; ++c16) {
            const int chunk = ((qc & 63) >> 3) + c16;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(dk[4 * c16], dk[4 * c16 + 1], dk[4 * c16 + 2], dk[4 * c16 + 3]);
          }
        }
        fence_async_shared();
        tc_fence_before();
        FA_PAIR_REPORT(&bar->ew_done, lead_ew_done);
      }
      // ---- epilogue: warpgroup 0 writes dK = scale dK_acc, warpgroup 1 dV
      if (!alive || !__all_sync(0xffffffffu, wait_bounded_cluster_inl(&bar->acc_done, w & 1, ctx, kSitePairAcc))) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t tAcc = tmem + (grp ? C::kDvCol : C::kDkCol) + lane_off;
      const float mul = grp ? 1.f : p.scale;
      const int kg = t.jb * 128 + r;
      __nv_bfloat16* out = (grp ? p.dv_out : p.dk_out) + ((size_t)t.bh * N + kg) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tAcc + 32 * c, v);
        tmem_wait_ld();
        reg_fence32(v);
        if (kg < N) {
          uint32_t w16[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2)
            w16[e2] = pack_bf16x2(__uint_as_float(v[2 * e2]) * mul, __uint_as_float(v[2 * e2 + 1]) * mul);
          if (p.out_align32) {
            st_global_v8(out + 32 * c, w16);
            st_global_v8(out + 32 * c + 16, w16 + 8);
          } else {
            uint4* o4 = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              o4[v4] = make_uint4(w16[4 * v4], w16[4 * v4 + 1], w16[4 * v4 + 2], w16[4 * v4 + 3]);
          }
        }
      }
      tc_fence_before();
    }
#undef FA_PAIR_REPORT
  }

  tc_fence_before();
  __syncthreads();
  // the leader's products (which read the peer's shared and tensor memory) have
  // completed, and neither CTA touches the other's memory after this
  cluster_sync();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

}  // namespace fa
