// Deterministic dQ: a separate, query-major pass of the backward.
//
// "Interrogating the GPU part 5: FlashAttention", "What does the backward
// pass do without P?": every probability tile is recomputed from Q, K and the
// saved log-sum-exp, P_ij = exp(S_ij - L_i), and dS = P o (dP - delta) with
// dP = dO V^T; then dQ = scale dS K.  "LLM Flash Attention", "End-to-end
// flow" (backward paragraph): the gradients come from the recomputed tiles.
//
// The main backward kernel works per key block and can only add its share of
// dQ_i into a shared fp32 accumulator with atomics, whose order (and hence
// rounding) changes from run to run.  This kernel instead owns one query
// block i of one (batch, head) and visits the key blocks j in a fixed order,
// recomputing
//   S  = Q_i K_j^T,  dP = dO_i V_j^T               (issuer A, fp32 in TMEM)
//   P  = 2^(S scale log2e - L_i log2e), masked on the causal diagonal,
//   dS = P o (dP - delta_i)                        (elementwise warps, bf16 to smem)
//   dQ += dS K_j                                    (issuer B, fp32 in TMEM)
// and writes dQ = scale dQ once, so the result is bitwise repeatable.  It
// costs three products per tile (two of them repeated from the main kernel).
//
// Warp roles (384 threads):
//   warps 0-3  elementwise, key columns 0-63 of every block (thread = query row)
//   warps 4-7  elementwise, key columns 64-127
//   warp  8    issuer A (S, dP) and TMEM owner
//   warp  9    TMA producer: Q_i, dO_i once, then K_j and V_j in two rings
//   warp  10   issuer B (dQ)
//   warp  11   idle
// The elementwise warps copy S and dP into registers and release the tensor
// memory at once, so the next block's S and dP are computed while they work.
// Tensor memory: S at column 0, dP at 128, dQ at 256.  Shared memory: Q_i,
// dO_i, the bf16 dS tile (queries x keys, K-major for the dQ product), and
// the K and V rings; all tiles 128-byte swizzled.
#pragma once

#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

template <int D>
struct BwdDqCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kAtoms = D / 64;
  static constexpr int kKSlots = (D == 128) ? 2 : 4;
  static constexpr int kVSlots = (D == 128) ? 2 : 4;
  static constexpr int kDsBytes = 128 * 128 * 2;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSCol = 0, kDpCol = 128, kDqCol = 256;
  // dynamic shared memory is declared 1024-byte aligned (checked at run time)
  static constexpr int kSmemBytes = 2 * kTileBytes + kDsBytes + (kKSlots + kVSlots) * kTileBytes + 256;
};

struct BwdDqBarriers {
  uint64_t qd_full;
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full, s_free, dp_full, dp_free, ds_full, ds_free, acc_done;
  uint64_t drain[2];
  uint64_t never;
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(BwdDqBarriers) <= 256, "barriers overflow their shared-memory slot");

struct BwdDqParams {
  const float* delta_pad;  // [B*H][Npad] delta, 0 past N
  const float* lse2_pad;   // [B*H][Npad] LSE * log2(e), +inf past N
  __nv_bfloat16* dq;
  int N;
  int nqb;           // query (and key) blocks per head
  int num_bh;        // batch * heads
  int group_heads;   // with the mask: heads per group of the item order
  float scale_log2;  // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
  int debug_stall;
};

enum : int { kSiteDqProducer = 32, kSiteDqQ, kSiteDqK, kSiteDqV, kSiteDqSFree, kSiteDqDpFree, kSiteDqS, kSiteDqDp,
             kSiteDqDsFree, kSiteDqDs, kSiteDqAcc };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                     const BwdDqParams p) {
  using C = BwdDqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(&g_fa_device_status, 0u, kStatusBadSmem);
    return;
  }
  uint8_t* sQ = smem_raw;
  uint8_t* sDO = sQ + C::kTileBytes;
  uint8_t* sDS = sDO + C::kTileBytes;
  uint8_t* sK = sDS + C::kDsBytes;
  uint8_t* sV = sK + C::kKSlots * C::kTileBytes;
  BwdDqBarriers* bar = reinterpret_cast<BwdDqBarriers*>(sV + C::kVSlots * C::kTileBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  // query blocks from the last (the most key blocks when causal) to the
  // first: without the mask head by head; with it in groups of group_heads
  // heads, by query block first inside a group (the costliest block of every
  // head of the group, then the next), so that the hardware hands the
  // costliest CTAs out first while a group's K and V still fit in L2
  int ib, bh;
  if (CAUSAL) {
    const int per_group = p.group_heads * p.nqb;
    const int grp = (int)blockIdx.x / per_group;
    const int r = (int)blockIdx.x - grp * per_group;
    const int gh = min(p.group_heads, p.num_bh - grp * p.group_heads);
    ib = p.nqb - 1 - r / gh;
    bh = grp * p.group_heads + r % gh;
  } else {
    ib = p.nqb - 1 - (int)(blockIdx.x % p.nqb);
    bh = (int)(blockIdx.x / p.nqb);
  }
  const int q0 = ib * 128;
  const int nb = CAUSAL ? ib + 1 : p.nqb;  // key blocks visited

  if (tid == 0) {
    mbar_init(&bar->qd_full, 1);
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->k_empty[s], 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) {
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->v_empty[s], 1);
    }
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->s_free, 256);
    mbar_init(&bar->dp_full, 1);
    mbar_init(&bar->dp_free, 256);
    mbar_init(&bar->ds_full, 256);
    mbar_init(&bar->ds_free, 1);
    mbar_init(&bar->acc_done, 1);
    mbar_init(&bar->drain[0], 1);
    mbar_init(&bar->drain[1], 1);
    mbar_init(&bar->never, 1);
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(&bar->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) {
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_k);
    tma_prefetch_map(&map_v);
    tma_prefetch_map(&map_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtx ctx{&bar->abort_flag, p.wait_limit_ns};

  if (warp == 9) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar->qd_full, 2 * C::kTileBytes);
      for (int a = 0; a < C::kAtoms; ++a) {
        tma_load_3d(sQ + a * 16384, &map_q, &bar->qd_full, a * 64, q0, bh);
        tma_load_3d(sDO + a * 16384, &map_do, &bar->qd_full, a * 64, q0, bh);
      }
      int nk = 0, nv = 0;
      bool ok = true;
      for (int j = 0; ok && j < nb; ++j) {
        {
          const int s = nk % C::kKSlots;
          if (!wait_bounded(&bar->k_empty[s], ((nk / C::kKSlots) & 1) ^ 1, ctx, kSiteDqProducer)) break;
          mbar_arrive_expect_tx(&bar->k_full[s], C::kTileBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sK + s * C::kTileBytes + a * 16384, &map_k, &bar->k_full[s], a * 64, j * 128, bh);
          ++nk;
        }
        {
          const int s = nv % C::kVSlots;
          if (!wait_bounded(&bar->v_empty[s], ((nv / C::kVSlots) & 1) ^ 1, ctx, kSiteDqProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar->v_full[s], C::kTileBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sV + s * C::kTileBytes + a * 16384, &map_v, &bar->v_full[s], a * 64, j * 128, bh);
          ++nv;
        }
      }
      // every copy this thread started must land before the CTA can exit
      wait_drain(&bar->qd_full, 0, kDrainLimitNs);
      for (int s = 0; s < C::kKSlots; ++s)
        if (nk > s) wait_drain(&bar->k_full[s], ((nk - 1 - s) / C::kKSlots) & 1, kDrainLimitNs);
      for (int s = 0; s < C::kVSlots; ++s)
        if (nv > s) wait_drain(&bar->v_full[s], ((nv - 1 - s) / C::kVSlots) & 1, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ------------------------------------------------------------------ issuer A: S and dP
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dodesc = sdesc_sw128(smem_u32(sDO), 16, 1024);
      bool ok = !(p.debug_stall && !wait_bounded(&bar->never, 0, ctx, kSiteStall));
      ok = ok && wait_bounded(&bar->qd_full, 0, ctx, kSiteDqQ);
      for (int j = 0; ok && j < nb; ++j) {
        // S = Q_i K_j^T once the elementwise warps have copied the previous S out
        const int ks = j % C::kKSlots;
        if (!wait_bounded(&bar->k_full[ks], (j / C::kKSlots) & 1, ctx, kSiteDqK)) break;
        if (j > 0 && !wait_bounded(&bar->s_free, (j - 1) & 1, ctx, kSiteDqSFree)) break;
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK + ks * C::kTileBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + C::kSCol, qdesc + off, kdesc + off, id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar->s_full);
        // dP = dO_i V_j^T once the previous dP has been copied out; V_j is then done
        const int vs = j % C::kVSlots;
        if (!wait_bounded(&bar->v_full[vs], (j / C::kVSlots) & 1, ctx, kSiteDqV)) break;
        if (j > 0 && !wait_bounded(&bar->dp_free, (j - 1) & 1, ctx, kSiteDqDpFree)) break;
        tc_fence_after();
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV + vs * C::kTileBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + C::kDpCol, dodesc + off, vdesc + off, id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar->dp_full);
        mma_commit(&bar->v_empty[vs]);
      }
      mma_commit(&bar->drain[0]);
      wait_drain(&bar->drain[0], 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------------ issuer B: dQ
    if (lane == 0) {
      // A = dS (queries x keys, K-major), B = K_j (keys x d, read N-major)
      constexpr uint32_t id_q = idesc_bf16_f32(128, D, false, true);
      const uint64_t dsdesc = sdesc_sw128(smem_u32(sDS), 16, 1024);
      bool ok = true;
      int j = 0;
      for (; ok && j < nb; ++j) {
        if (!wait_bounded(&bar->ds_full, j & 1, ctx, kSiteDqDs)) break;
        tc_fence_after();
        const int ks = j % C::kKSlots;
        const uint64_t kdesc_mn = sdesc_sw128(smem_u32(sK + ks * C::kTileBytes), 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + C::kDqCol, dsdesc + aoff, kdesc_mn + (uint32_t)((kk * 2048) >> 4), id_q,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        // dS and K_j have been read once these products complete
        mma_commit(&bar->ds_free);
        mma_commit(&bar->k_empty[ks]);
      }
      if (j == nb) mma_commit(&bar->acc_done);
      mma_commit(&bar->drain[1]);
      wait_drain(&bar->drain[1], 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------------ elementwise
    const int g = warp >> 2;   // key columns [64 g, 64 g + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row in the block
    const int row_g = q0 + r;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + C::kSCol + lane_off + 64 * g;
    const uint32_t tDP = tmem + C::kDpCol + lane_off + 64 * g;
    const size_t stat_row = (size_t)bh * (p.nqb * 128) + row_g;  // padded statistics
    const float nl2 = -__ldg(p.lse2_pad + stat_row);              // -inf past N: P = 0 there
    const float delta = __ldg(p.delta_pad + stat_row);
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    const float2 nl2_2 = make_float2(nl2, nl2);
    const float2 nd2 = make_float2(-delta, -delta);
    uint8_t* ds_row = sDS + g * 16384 + r * 128;
    bool alive = true;
    for (int j = 0; alive && j < nb; ++j) {
      // P = 2^(S c - L log2e) for this warpgroup's 64 keys, S released at once
      if (!__all_sync(0xffffffffu, wait_bounded(&bar->s_full, j & 1, ctx, kSiteDqS))) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(tS, sv[0]);
      tmem_ld32(tS + 32, sv[1]);
      tmem_wait_ld();
      reg_fence32(sv[0]);
      reg_fence32(sv[1]);
      tc_fence_before();
      mbar_arrive(&bar->s_free);
      float2 pf[32];
      const bool diag = CAUSAL && (j == ib);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[h][2 * e]), __uint_as_float(sv[h][2 * e + 1])),
                                      c2, nl2_2);
          float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (diag) {  // key 128 j + c is in the future of query row_g when c > r
            const int c = 64 * g + 32 * h + 2 * e;
            if (c > r) pe.x = 0.f;
            if (c + 1 > r) pe.y = 0.f;
          }
          pf[16 * h + e] = pe;
        }
      }
      // dS = P o (dP - delta), dP released at once
      if (!__all_sync(0xffffffffu, wait_bounded(&bar->dp_full, j & 1, ctx, kSiteDqDp))) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t dv[2][32];
      tmem_ld32(tDP, dv[0]);
      tmem_ld32(tDP + 32, dv[1]);
      tmem_wait_ld();
      reg_fence32(dv[0]);
      reg_fence32(dv[1]);
      tc_fence_before();
      mbar_arrive(&bar->dp_free);
      uint32_t dsk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 dpd =
              __fadd2_rn(make_float2(__uint_as_float(dv[h][2 * e]), __uint_as_float(dv[h][2 * e + 1])), nd2);
          const float2 dse = __fmul2_rn(pf[16 * h + e], dpd);
          dsk[16 * h + e] = pack_bf16x2(dse.x, dse.y);
        }
      }
      // the dS tile is free once the previous dQ product has read it
      if (j > 0 && !__all_sync(0xffffffffu, wait_bounded(&bar->ds_free, (j - 1) & 1, ctx, kSiteDqDsFree))) {
        alive = false;
        break;
      }
      // row r of atom g: 64 keys = 8 chunks of 16 B, chunk c at c ^ (r mod 8)
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4*>(ds_row + ((c16 ^ (r & 7)) << 4)) =
            make_uint4(dsk[4 * c16], dsk[4 * c16 + 1], dsk[4 * c16 + 2], dsk[4 * c16 + 3]);
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(&bar->ds_full);
    }
    // epilogue: dQ = scale dQ_acc -> bf16; warpgroup g writes columns [g D/2, (g+1) D/2) of its rows
    if (alive && __all_sync(0xffffffffu, wait_bounded(&bar->acc_done, 0, ctx, kSiteDqAcc))) {
      tc_fence_after();
      __nv_bfloat16* out = p.dq + ((size_t)bh * N + row_g) * D + g * (D / 2);
      const float sc = p.scale;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + C::kDqCol + lane_off + g * (D / 2) + 32 * c, v);
        tmem_wait_ld();
        reg_fence32(v);
        if (row_g < N) {
          uint4* o4 = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * v4 + 0]) * sc, __uint_as_float(v[8 * v4 + 1]) * sc);
            w.y = pack_bf16x2(__uint_as_float(v[8 * v4 + 2]) * sc, __uint_as_float(v[8 * v4 + 3]) * sc);
            w.z = pack_bf16x2(__uint_as_float(v[8 * v4 + 4]) * sc, __uint_as_float(v[8 * v4 + 5]) * sc);
            w.w = pack_bf16x2(__uint_as_float(v[8 * v4 + 6]) * sc, __uint_as_float(v[8 * v4 + 7]) * sc);
            o4[v4] = w;
          }
        }
      }
    }
  }
  // warp 11 has no role

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
