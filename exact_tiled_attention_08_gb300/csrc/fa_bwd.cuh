// Backward kernels.
//
// "Interrogating the GPU part 5: FlashAttention", "What does the backward
// pass do without P?": the forward pass keeps one log-sum-exp per row, and
// the backward pass recomputes every probability tile P_ij = exp(S_ij - L_i)
// from Q, K and L, then forms dV = P^T dO and dS = P o (dP - delta).
#pragma once

#include <cuda_bf16.h>

#include <math_constants.h>

#include "sm103_ptx.cuh"

namespace fa {

// ---------------------------------------------------------------------------
// preprocess: delta_i = sum_c dO_ic O_ic (fp32), and optionally zero the fp32
// dQ accumulator rows.  Memory-bound: one 16-byte load of O and of dO per
// thread per row; D/8 threads per row.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
    fa_bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                             float* __restrict__ delta, float* __restrict__ dq_acc, long long rows) {
  constexpr int kThreadsPerRow = D / 8;
  constexpr int kRowsPerPass = 256 / kThreadsPerRow;
  const int sub = threadIdx.x % kThreadsPerRow;
  const int rloc = threadIdx.x / kThreadsPerRow;
  for (long long base = (long long)blockIdx.x * kRowsPerPass; base < rows;
       base += (long long)gridDim.x * kRowsPerPass) {
    const long long row = base + rloc;
    const bool valid = row < rows;
    float s = 0.f;
    if (valid) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + sub);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa2 = __bfloat1622float2(a2[i]);
        const float2 fb2 = __bfloat1622float2(b2[i]);
        s = fmaf(fa2.x, fb2.x, s);
        s = fmaf(fa2.y, fb2.y, s);
      }
    }
#pragma unroll
    for (int off = kThreadsPerRow / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (valid) {
      if (sub == 0) delta[row] = s;
      if (dq_acc) {
        float4* z = reinterpret_cast<float4*>(dq_acc + row * D) + 2 * sub;
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// preprocess of fa_bwd: per row of each (batch, head), padded to a whole
// number of 128-row blocks (Npad = 128 ceil(N / 128)):
//   delta_pad[bh][n] = sum_c dO_nc O_nc      (0 for n >= N)
//   lse2_pad[bh][n]  = LSE_n * log2(e)       (+inf for n >= N, so P = 0 there)
// and the fp32 dQ accumulator rows are zeroed (when there is one).  The padded, 128-aligned rows
// let the main kernel bring both vectors in with TMA next to each Q tile.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                       const float* __restrict__ lse, float* __restrict__ delta_pad, float* __restrict__ lse2_pad,
                       float* __restrict__ dq_acc, int N, int Npad, long long padded_rows) {
  constexpr int kThreadsPerRow = D / 8;
  constexpr int kRowsPerPass = 256 / kThreadsPerRow;
  const int sub = threadIdx.x % kThreadsPerRow;
  const int rloc = threadIdx.x / kThreadsPerRow;
  for (long long base = (long long)blockIdx.x * kRowsPerPass; base < padded_rows;
       base += (long long)gridDim.x * kRowsPerPass) {
    const long long prow = base + rloc;  // padded row index bh * Npad + n
    const long long bh = prow / Npad;
    const int n = (int)(prow - bh * Npad);
    const bool in_range = prow < padded_rows;
    const bool valid = in_range && n < N;
    const long long row = bh * N + n;  // unpadded row
    float s = 0.f;
    if (valid) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + sub);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa2 = __bfloat1622float2(a2[i]);
        const float2 fb2 = __bfloat1622float2(b2[i]);
        s = fmaf(fa2.x, fb2.x, s);
        s = fmaf(fa2.y, fb2.y, s);
      }
    }
#pragma unroll
    for (int off = kThreadsPerRow / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (in_range && sub == 0) {
      delta_pad[prow] = valid ? s : 0.f;
      lse2_pad[prow] = valid ? __ldg(lse + row) * 1.4426950408889634f : CUDART_INF_F;
    }
    if (valid && dq_acc) {
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D) + 2 * sub;
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// main backward kernel: the work is one item per (key block j, batch, head).
// With the causal mask one CTA runs per item (the items' costs range from 1
// to nkb query blocks; bwd_item hands the costliest out first and the
// hardware's CTA scheduler balances them); without it the CTAs are
// persistent, one per SM, and walk the items blockIdx.x, blockIdx.x +
// gridDim.x, ...  All pipeline counters (slot uses, per-block barrier
// phases, statistics entries) run on across the items: a CTA loads the next
// item's K and V, then its first Q tile, as soon as the current item's last
// dK and dQ products have read the old K and V, and the reducers' last dQ_i
// and the dK, dV write-out overlap with the next item's first products.
//
// K_j and V_j (128 keys) stay in shared memory; the query blocks i (all of
// them, or i >= j when causal) stream Q_i (with its rows' LSE log2(e) and
// delta) and dO_i through slots of their own (BwdCfg).  Per query block, in the transposed
// orientation (TMEM lane = key, column = query):
//   S^T = K_j Q_i^T, then dP^T = V_j dO_i^T      (issuer A)
//   P^T  = 2^(S^T scale log2e - LSE_i log2e), masked on the causal diagonal
//                                                  (elementwise warps, thread = key)
//   dV += P^T dO_i                                 (issuer B, as soon as P^T is written)
//   dS^T = P^T o (dP^T - delta_i)                  (elementwise warps)
//   dQ_i = dS K_j, then dK += dS^T Q_i            (issuer B)
// and the reducer warps add dQ_i into the fp32 accumulator in global memory
// while the next query block is processed.  The elementwise step is split in
// two so that dV runs while dS^T is computed, and the next block's S^T (whose
// columns dV frees) while dK and dQ run.  dK, dV accumulate in TMEM across
// the item's query blocks and are written once at the end of the item.
//
// The global fp32 reduction of dQ_i (64 KB per query block at d = 128) takes
// about as long as the rest of a query block; it therefore runs on warps of
// its own that hold dQ_i in registers, so that TMEM is free for the next dP^T
// at once and the elementwise warps never wait for it, and it goes through
// TMA reduces, off the load/store path the elementwise warps' shared-memory
// stores use.
//
// Warp roles (512 threads, four warpgroups; register budgets set with
// setmaxnreg, 136 + 136 + 152 + 88 per thread = the launch's 128 x 4):
//   warps 0-7   elementwise: warpgroup g owns query columns [64 g, 64 g + 64)
//               of dS
//   warps 8-11  reducers: warp 8 + q takes TMEM lanes 32q.. (query rows) of
//               dQ_i into registers, releases the columns, writes 32 x 32
//               blocks into two 4 KB tiles of its own in the TMA's swizzled
//               layout and adds each to the accumulator with one TMA reduce
//   warp  12    issuer A (S^T and dP^T) and TMEM owner
//   warp  13    TMA producer: K, V and the Q tiles
//   warp  14    issuer B (dV, dQ and dK)
//   warp  15    TMA producer: the dO tiles
// Tensor memory: dK at column 0, dV at d, S^T at 2d, dP^T at 2d + 128.  The
// bf16 P^T of query group G (queries 16G..16G+15) is written over the first 8
// of that group's own S^T columns, which only the writing thread has read;
// dQ_i goes into the dP^T columns once the elementwise step has read them.
// ---------------------------------------------------------------------------
// Register budgets per thread after setmaxnreg: the two elementwise
// warpgroups take BwdRegs::kWork, the reducers kRed (a reducer holds its
// 32 rows of dQ_i, D values each, in registers), the issuing/producer
// warpgroup keeps kMisc.  Each SM sub-partition holds one warp of
// every warpgroup, so 2 x 136 + 152 + 88 = 512 = 4 x 128 uses exactly the
// registers the block was launched with (128 per thread, which the host
// checks before launching).
// At d = 64 a reducer's rows are half as long, and the elementwise warps,
// which set the pace there, take 160 (2 x 160 + 104 + 88 = 512; the reducers
// then give registers back).  Without the atomic dQ the reducer warpgroup
// has no role and keeps the launch budget (2 x 136 + 128 + 88 < 512).
// setmaxnreg.inc only raises a warp's count and .dec only lowers it.
template <int D, bool kAtomicDq>
struct BwdRegs {
  static constexpr uint32_t kLaunch = 128, kMisc = 88;
  static constexpr uint32_t kWork = (D == 64 && kAtomicDq) ? 160 : 136;
  static constexpr uint32_t kRed = kAtomicDq ? 4 * kLaunch - 2 * kWork - kMisc : kLaunch;
  static_assert(2 * kWork + kRed + kMisc <= 4 * kLaunch, "register split must fit the launch budget");
  static_assert(kWork > kLaunch && kMisc < kLaunch, "the elementwise warps raise, the issuing warps lower");
  static_assert(kWork % 8 == 0 && kWork <= 256 && kRed % 8 == 0 && kRed >= 24 && kRed <= 256 && kMisc % 8 == 0 &&
                    kMisc >= 24,
                "setmaxnreg takes multiples of 8 in [24, 256]");
};

// kAtomicDq: the kernel also forms dQ_i = dS K_j and adds it into the fp32
// accumulator (reducer warps); otherwise dQ is left to the separate
// deterministic pass, and the shared memory of the reducers' staging tiles
// goes to a fourth tile slot (a second dO slot) at d = 128.
template <int D, bool kAtomicDq>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kAtoms = D / 64;
  static constexpr int kSlots = (D == 128) ? (kAtomicDq ? 3 : 4) : 6;   // Q and dO tiles
  // Q tiles and dO tiles have slots of their own: Q_g goes to Q slot
  // g % kQSlots once dK of block g - kQSlots has released it, dO_g to dO slot
  // g % kDoSlots once dV of block g - kDoSlots has.  dV runs right after the
  // first half of the elementwise step, so with three slots (two for Q, one
  // for dO) the next dO tile loads while the second half and dQ, dK run, and
  // the next Q tile is a whole block ahead.
  static constexpr int kQSlots = (kSlots + 1) / 2, kDoSlots = kSlots / 2;
  // LSE*log2e [128] and delta [128] of a query block come with its Q tile; the
  // entry of block g is reused by block g + kQSlots, whose Q loads once dK of
  // block g, which follows its elementwise step, has run
  static constexpr int kStatBytes = 1024;
  static constexpr int kStatEntries = kQSlots;
  static constexpr int kDsBytes = 128 * 128 * 2;      // dS^T tile: 2 atom columns of 64 queries
  // reducers: two 32 x 32 fp32 tiles per warp, each added to the accumulator
  // by one TMA reduce while the warp fills the other
  static constexpr int kStageBytes = kAtomicDq ? 4 * 2 * 4096 : 0;
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;             // 65536 / 512
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kDkCol = 0, kDvCol = D, kSCol = 2 * D, kDpCol = 2 * D + 128;
  // the dynamic shared memory is declared 1024-byte aligned (checked at run
  // time), so no alignment slack is added
  static constexpr int kSmemBytes =
      2 * kTileBytes + kSlots * kTileBytes + kDsBytes + kStageBytes + kStatEntries * kStatBytes + 256;
};

struct BwdBarriers {
  uint64_t kv_full;
  uint64_t ring_full[8];
  uint64_t ring_empty[8];
  uint64_t s_full, dp_full, p_done, ew_done, dv_done, dq_full, dq_free, dk_done, acc_done;
  uint64_t drain[2];
  uint64_t never;  // signalled by nothing: the debug stall waits on it
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(BwdBarriers) <= 256, "barriers overflow their shared-memory slot");

struct BwdParams {
  float* dq_acc;  // [B*H][N][d] fp32, zeroed by the preprocess
  __nv_bfloat16* dk_out;
  __nv_bfloat16* dv_out;
  int N;
  int nkb;           // key (and query) blocks per head
  int num_items;     // (key block, batch, head) items: nkb * batch * heads
  int num_bh;        // batch * heads
  int group_heads;   // with the mask: heads per group of the item order (see bwd_item)
  float scale_log2;  // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
  int debug_stall;  // nonzero: issuer A first waits on `never` (tests the timeout path)
  int out_align32;  // nonzero: dk_out and dv_out are 32-byte aligned (32-byte stores)
};

// The CTA's items: blockIdx.x, blockIdx.x + gridDim.x, ...
// Without the mask item k is key block k % nkb of (batch, head) k / nkb, so
// that the CTAs running at one time work on few heads, whose Q and dO tiles
// they share through L2.  With the mask item j costs nkb - j query blocks;
// the items go in groups of group_heads heads, and inside a group by key
// block first (j = 0, the costliest, for every head of the group, then
// j = 1, ...): the hardware hands the costliest items out first, so that the
// last SMs to finish end on one-block items, while a group's Q and dO still
// fit in L2.
struct BwdItem {
  int bh, jb, i_start, n_it;
};
template <bool CAUSAL>
__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int k) {
  BwdItem t;
  if (CAUSAL) {
    const int per_group = p.group_heads * p.nkb;
    const int grp = k / per_group;
    const int r = k - grp * per_group;
    const int gh = min(p.group_heads, p.num_bh - grp * p.group_heads);  // heads in this group
    t.jb = r / gh;
    t.bh = grp * p.group_heads + (r - t.jb * gh);
  } else {
    t.bh = k / p.nkb;
    t.jb = k - t.bh * p.nkb;
  }
  t.i_start = CAUSAL ? t.jb : 0;
  t.n_it = p.nkb - t.i_start;
  return t;
}

enum : int { kSiteBwdProducer = 16, kSiteBwdKV, kSiteBwdQ, kSiteBwdDo, kSiteBwdDvDone, kSiteBwdDqFree, kSiteBwdEw,
             kSiteBwdS, kSiteBwdDp, kSiteBwdDq, kSiteBwdAcc };

template <int D, bool CAUSAL, bool kAtomicDq>
__global__ void __launch_bounds__(512, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_lse2, const __grid_constant__ CUtensorMap map_delta,
                  const __grid_constant__ CUtensorMap map_dq, const BwdParams p) {
  using C = BwdCfg<D, kAtomicDq>;
  static_assert(BwdRegs<D, kAtomicDq>::kLaunch == C::kLaunchRegs, "register split of the launch budget");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    // the 128-byte-swizzled tiles need 1024-byte alignment: report, do nothing
    if (threadIdx.x == 0) atomicCAS(&g_fa_device_status, 0u, kStatusBadSmem);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTileBytes;
  uint8_t* sRing = smem + 2 * C::kTileBytes;
  uint8_t* sDS = sRing + C::kSlots * C::kTileBytes;
  uint8_t* sStage = sDS + C::kDsBytes;
  // query block g: entry g % kStatEntries = LSE*log2e [128], delta [128]
  uint8_t* sStat = sStage + C::kStageBytes;
  BwdBarriers* bar = reinterpret_cast<BwdBarriers*>(sStat + C::kStatEntries * C::kStatBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;

  if (tid == 0) {
    mbar_init(&bar->kv_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar->ring_full[s], 1);
      mbar_init(&bar->ring_empty[s], 1);
    }
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->dp_full, 1);
    mbar_init(&bar->p_done, 256);
    mbar_init(&bar->ew_done, 256);
    mbar_init(&bar->dv_done, 1);
    mbar_init(&bar->dq_full, 1);
    mbar_init(&bar->dq_free, 128);
    mbar_init(&bar->dk_done, 1);
    mbar_init(&bar->acc_done, 1);
    mbar_init(&bar->drain[0], 1);
    mbar_init(&bar->drain[1], 1);
    mbar_init(&bar->never, 1);
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(&bar->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_k);
    tma_prefetch_map(&map_v);
    tma_prefetch_map(&map_do);
    tma_prefetch_map(&map_lse2);
    tma_prefetch_map(&map_delta);
    if (kAtomicDq) tma_prefetch_map(&map_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtx ctx{&bar->abort_flag, p.wait_limit_ns};
  if (warp >= 12) {
    setmaxnreg_dec<BwdRegs<D, kAtomicDq>::kMisc>();
    if (warp == 13 || warp == 15) {
      // ---------------------------------------------------------------- TMA producers
      // warp 13: K and V of each item and the Q tiles (with the statistics),
      // warp 15: the dO tiles, so that neither queue waits on the other's
      // slot.  g counts query blocks over all of the CTA's items.
      if (lane == 0) {
        const bool q_side = warp == 13;
        const int nslot = q_side ? C::kQSlots : C::kDoSlots, slot0 = q_side ? 0 : C::kQSlots;
        int g = 0, w = 0, kv_loads = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x, ++w) {
          const BwdItem t = bwd_item<CAUSAL>(p, item);
          if (q_side) {
            // K and V of the item, once the previous item's last products
            // (acc_done) have read the old ones
            if (w > 0 && !wait_bounded_inl(&bar->acc_done, (w - 1) & 1, ctx, kSiteBwdProducer)) break;
            mbar_arrive_expect_tx(&bar->kv_full, 2 * C::kTileBytes);
            for (int a = 0; a < C::kAtoms; ++a) {
              tma_load_3d(sK + a * 16384, &map_k, &bar->kv_full, a * 64, t.jb * 128, t.bh);
              tma_load_3d(sV + a * 16384, &map_v, &bar->kv_full, a * 64, t.jb * 128, t.bh);
            }
            ++kv_loads;
          }
          for (int it = 0; it < t.n_it; ++it, ++g) {
            const int i = t.i_start + it;
            const int s = slot0 + g % nslot;
            if (!wait_bounded_inl(&bar->ring_empty[s], ((g / nslot) & 1) ^ 1, ctx, kSiteBwdProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bar->ring_full[s], C::kTileBytes + (q_side ? C::kStatBytes : 0));
            const CUtensorMap* map = q_side ? &map_q : &map_do;
            for (int a = 0; a < C::kAtoms; ++a)
              tma_load_3d(sRing + s * C::kTileBytes + a * 16384, map, &bar->ring_full[s], a * 64, i * 128, t.bh);
            if (q_side) {
              uint8_t* st = sStat + (g % C::kStatEntries) * C::kStatBytes;
              tma_load_2d(st, &map_lse2, &bar->ring_full[s], i * 128, t.bh);
              tma_load_2d(st + 512, &map_delta, &bar->ring_full[s], i * 128, t.bh);
            }
          }
        }
        // every load this warp started has landed before the CTA may end
        if (kv_loads > 0) wait_drain_inl(&bar->kv_full, (kv_loads - 1) & 1, kDrainLimitNs);
        for (int k = 0; k < nslot; ++k) {
          if (g > k) {
            const int uses = (g - 1 - k) / nslot + 1;
            wait_drain_inl(&bar->ring_full[slot0 + k], (uses - 1) & 1, kDrainLimitNs);
          }
        }
      }
      __syncwarp();
    } else if (warp == 12) {
      // ---------------------------------------------------------------- issuer A: S^T and dP^T
      if (lane == 0) {
        constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
        const uint32_t ring = smem_u32(sRing);
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint32_t tS = tmem + C::kSCol, tDP = tmem + C::kDpCol;
        bool ok = !(p.debug_stall && !wait_bounded_inl(&bar->never, 0, ctx, kSiteStall));
        // S^T goes first: the first half of the elementwise step needs only
        // S^T, its columns are free as soon as dV of the previous block has
        // run, and dP^T waits for the reducers to take the previous dQ out of
        // its columns.
        // g counts query blocks over all of the CTA's items, w the items.
        int g = 0, w = 0;
        for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x, ++w) {
          const BwdItem t = bwd_item<CAUSAL>(p, item);
          ok = wait_bounded_inl(&bar->kv_full, w & 1, ctx, kSiteBwdKV);
          for (int it = 0; ok && it < t.n_it; ++it, ++g) {
#pragma unroll
            for (int step = 0; step < 2; ++step) {
              if (step == 0) {
                // S^T = K Q_i^T, once dV has consumed the previous P^T held in
                // these columns
                const int sq = g % C::kQSlots;
                if (!wait_bounded_inl(&bar->ring_full[sq], (g / C::kQSlots) & 1, ctx, kSiteBwdQ)) {
                  ok = false;
                  break;
                }
                if (g > 0 && !wait_bounded_inl(&bar->dv_done, (g - 1) & 1, ctx, kSiteBwdDvDone)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t qdesc = sdesc_sw128(ring + sq * C::kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                  mma_bf16_ss(tS, kdesc + off, qdesc + off, id_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar->s_full);
              } else {
                // dP^T = V dO_i^T, once the reducers have taken the previous dQ
                // out of these columns (without dQ: once the elementwise step
                // has read the previous dP^T)
                const int sd = C::kQSlots + g % C::kDoSlots;
                if (!wait_bounded_inl(&bar->ring_full[sd], (g / C::kDoSlots) & 1, ctx, kSiteBwdDo)) {
                  ok = false;
                  break;
                }
                if (g > 0 && !wait_bounded_inl(kAtomicDq ? &bar->dq_free : &bar->ew_done, (g - 1) & 1, ctx,
                                               kSiteBwdDqFree)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t dodesc = sdesc_sw128(ring + sd * C::kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                  mma_bf16_ss(tDP, vdesc + off, dodesc + off, id_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar->dp_full);
              }
            }
          }
        }
        mma_commit(&bar->drain[0]);
        wait_drain_inl(&bar->drain[0], 0, kDrainLimitNs);
      }
      __syncwarp();
    } else if (warp == 14) {
      // ---------------------------------------------------------------- issuer B: dV, dQ and dK
      if (lane == 0) {
        constexpr uint32_t id_v = idesc_bf16_f32(128, D, false, true);  // dV (A = P^T in TMEM), dK
        constexpr uint32_t id_q = idesc_bf16_f32(128, D, true, true);   // dQ (A = dS, M-major)
        const uint32_t ring = smem_u32(sRing);
        const uint64_t kdesc_mn = sdesc_sw128(smem_u32(sK), 16384, 1024);
        const uint64_t dsdesc_k = sdesc_sw128(smem_u32(sDS), 16, 1024);
        const uint64_t dsdesc_mn = sdesc_sw128(smem_u32(sDS), 16384, 1024);
        const uint32_t tS = tmem + C::kSCol, tDP = tmem + C::kDpCol;
        const uint32_t tDK = tmem + C::kDkCol, tDV = tmem + C::kDvCol;
        bool ok = true;
        int g = 0;
        for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
          const BwdItem t = bwd_item<CAUSAL>(p, item);
          for (int it = 0; ok && it < t.n_it; ++it, ++g) {
            const int sq = g % C::kQSlots, sd = C::kQSlots + g % C::kDoSlots;
            // dV += P^T dO_i as soon as the elementwise warps have written P^T
            // (P^T of query group kk sits at S^T column 16 kk) and dP^T, which
            // also reads dO_i, is complete (so dO_i has landed, and its slot can
            // be released after dV); this frees the S^T columns for the next
            // block's scores
            ok = wait_bounded_inl(&bar->dp_full, g & 1, ctx, kSiteBwdEw) &&
                 wait_bounded_inl(&bar->p_done, g & 1, ctx, kSiteBwdEw);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dodesc_mn = sdesc_sw128(ring + sd * C::kTileBytes, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ts(tDV, tS + kk * 16, dodesc_mn + (uint32_t)((kk * 2048) >> 4), id_v,
                          (it > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bar->dv_done);
            mma_commit(&bar->ring_empty[sd]);
            // dQ_i = dS K (into the dP^T columns, read by now; the next dP^T
            // waits for the reducers to take it out), then dK += dS^T Q_i, once
            // dS^T is written
            if (!(ok = wait_bounded_inl(&bar->ew_done, g & 1, ctx, kSiteBwdEw))) break;
            tc_fence_after();
            // (fully unrolled: the MMAs are issued back to back; in a loop, a
            // 32-cycle MMA at d = 64 outruns its issue.  The issuing warps get
            // 88 registers for the unrolled descriptors.)
            if (kAtomicDq) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss(tDP, dsdesc_mn + (uint32_t)((kk * 2048) >> 4), kdesc_mn + (uint32_t)((kk * 2048) >> 4), id_q,
                            kk > 0 ? 1u : 0u);
              mma_commit(&bar->dq_full);
            }
            const uint64_t qdesc_mn = sdesc_sw128(ring + sq * C::kTileBytes, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
              mma_bf16_ss(tDK, dsdesc_k + off, qdesc_mn + (uint32_t)((kk * 2048) >> 4), id_v,
                          (it > 0 || kk > 0) ? 1u : 0u);
            }
            // Q_i has been read by S^T (long complete) and dK: release its slot;
            // the dS^T tile is free for the next elementwise step (dQ, issued
            // before dK, has read it too)
            mma_commit(&bar->ring_empty[sq]);
            mma_commit(&bar->dk_done);
          }
          // the item's dK and dV are complete, and its K and V read for the last time
          if (ok) mma_commit(&bar->acc_done);
        }
        mma_commit(&bar->drain[1]);
        wait_drain_inl(&bar->drain[1], 0, kDrainLimitNs);
      }
      __syncwarp();
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------------ reducers
    // (no role without the atomic dQ: the warpgroup keeps its launch budget)
    if (kAtomicDq) {
    using R = BwdRegs<D, kAtomicDq>;
    if constexpr (R::kRed > R::kLaunch)
      setmaxnreg_inc<R::kRed>();
    else if constexpr (R::kRed < R::kLaunch)
      setmaxnreg_dec<R::kRed>();
    const int q = warp & 3;
    const uint32_t tDQ = tmem + C::kDpCol + ((uint32_t)(q * 32) << 16);
    uint8_t* stage = sStage + q * 8192;  // two 4 KB tiles
    constexpr int kChunks = D / 32;      // 32-column chunks of a dQ row
    bool alive = true;
    int g = 0, r = 0;                    // r: tiles handed to the TMA so far
    for (int item = blockIdx.x; alive && item < p.num_items; item += gridDim.x) {
      const BwdItem t = bwd_item<CAUSAL>(p, item);
      for (int it = 0; it < t.n_it; ++it, ++g) {
        if (!__all_sync(0xffffffffu, wait_bounded_inl(&bar->dq_full, g & 1, ctx, kSiteBwdDq))) {
          alive = false;
          break;
        }
        tc_fence_after();
        uint32_t dqv[kChunks][32];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tmem_ld32(tDQ + 32 * c, dqv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kChunks; ++c) reg_fence32(dqv[c]);
        // dQ_i is in registers: issuer A may overwrite these columns with dP^T
        tc_fence_before();
        mbar_arrive(&bar->dq_free);
        // thread = query row 32 q + lane.  Each 32 x 32 block goes to a stage
        // tile in the TMA's 128-byte-swizzled layout (row = lane, 16-byte chunk
        // j at position j ^ (row & 7)), and one TMA reduce adds the tile to the
        // accumulator (rows past N are not written).  The two tiles alternate:
        // before a tile is refilled, the reduce issued from it two chunks ago
        // must have read it.
        const int qrow0 = (t.i_start + it) * 128 + 32 * q;
#pragma unroll
        for (int c = 0; c < kChunks; ++c, ++r) {
          uint8_t* tile = stage + (r & 1) * 4096;
          if (r >= 2) {
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
          }
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16)
            *reinterpret_cast<uint4*>(tile + lane * 128 + ((c16 ^ (lane & 7)) << 4)) =
                make_uint4(dqv[c][4 * c16], dqv[c][4 * c16 + 1], dqv[c][4 * c16 + 2], dqv[c][4 * c16 + 3]);
          fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            // (a tile wholly past N, in the last block of a head, is not sent;
            // its group is empty)
            if (qrow0 < N) tma_reduce_add_3d(&map_dq, tile, 32 * c, qrow0, t.bh);
            tma_store_commit();
          }
        }
      }
    }
    // every reduce has completed (and read its tile) before the CTA ends
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ elementwise
    setmaxnreg_inc<BwdRegs<D, kAtomicDq>::kWork>();
    const int grp = warp >> 2;  // warpgroup: query columns [64 grp, 64 grp + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + C::kSCol + lane_off;
    const uint32_t tDP = tmem + C::kDpCol + lane_off;
    const float sl2 = p.scale_log2;
    uint8_t* ds_row = sDS + grp * 16384 + r * 128;
    bool alive = true;
    int g = 0, w = 0;
    for (int item = blockIdx.x; alive && item < p.num_items; item += gridDim.x, ++w) {
      const BwdItem t = bwd_item<CAUSAL>(p, item);
      for (int it = 0; alive && it < t.n_it; ++it, ++g) {
        const float* stat = reinterpret_cast<const float*>(sStat + (g % C::kStatEntries) * C::kStatBytes);
        // ---- phase 1: P^T = 2^(S^T c - L log2e) into TMEM, the fp32 values kept
        // in registers; issuer B starts dV as soon as all of P^T is written
        if (!__all_sync(0xffffffffu, wait_bounded_inl(&bar->s_full, g & 1, ctx, kSiteBwdS))) {
          alive = false;
          break;
        }
        tc_fence_after();
        const bool diag = CAUSAL && it == 0;  // with the mask the first query block is i = j
        const float2 c2 = make_float2(sl2, sl2);
        float2 pf[2][16];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int qc = 64 * grp + 32 * ch;  // first query column of this chunk
          uint32_t sv[32];
          tmem_ld32(tS + qc, sv);
          tmem_wait_ld();
          reg_fence32(sv);
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            // four queries' L*log2e (the same for every thread: a broadcast read)
            const float4 l4 = *reinterpret_cast<const float4*>(stat + qc + 4 * e4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 4 * e4 + 2 * h;  // two queries at a time (packed fp32x2 arithmetic)
              const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
              const float2 xs = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nl);
              float2 pe = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
              if (diag) {  // key k0 + r is in the future of query qbase + qc + e
                if (qc + e < r) pe.x = 0.f;
                if (qc + e + 1 < r) pe.y = 0.f;
              }
              pf[ch][e / 2] = pe;
              pk[2 * e4 + h] = pack_bf16x2(pe.x, pe.y);
            }
          }
          // P^T of query groups qc/16 and qc/16 + 1 over the first 8 of their own columns
          tmem_st8(tS + qc, pk);
          tmem_st8(tS + qc + 16, pk + 8);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar->p_done);

        // ---- phase 2: dS^T = P^T o (dP^T - delta) into the shared dS^T tile,
        // once the previous block's dK and dQ have read it (dP^T of this block
        // was issued after the reducers took the previous dQ out of TMEM; dK,
        // which runs after dQ, reports on its own)
        bool ok2 = wait_bounded_inl(&bar->dp_full, g & 1, ctx, kSiteBwdDp);
        if (g > 0) ok2 = ok2 && wait_bounded_inl(&bar->dk_done, (g - 1) & 1, ctx, kSiteBwdDp);
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
              const int e = 4 * e4 + 2 * h;
              const float2 nd = h ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
              const float2 dpd = __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd);
              const float2 dse = __fmul2_rn(pf[ch][e / 2], dpd);
              dk[2 * e4 + h] = pack_bf16x2(dse.x, dse.y);
            }
          }
          // dS^T row r, queries [qc, qc+32): 4 chunks of 16 B in the swizzled atom grp
#pragma unroll
          for (int c16 = 0; c16 < 4; ++c16) {
            const int chunk = ((qc & 63) >> 3) + c16;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(dk[4 * c16], dk[4 * c16 + 1], dk[4 * c16 + 2], dk[4 * c16 + 3]);
          }
        }
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(&bar->ew_done);
      }
      // ---- epilogue: warpgroup 0 writes dK = scale dK_acc, warpgroup 1 writes
      // dV.  The next item's first dV and dK overwrite these columns only
      // after this warpgroup's next p_done arrival, which follows these reads.
      if (!alive || !__all_sync(0xffffffffu, wait_bounded_inl(&bar->acc_done, w & 1, ctx, kSiteBwdAcc))) {
        alive = false;
        break;
      }
      {
        tc_fence_after();
        const uint32_t tAcc = tmem + (grp ? C::kDvCol : C::kDkCol) + lane_off;
        const float mul = grp ? 1.f : p.scale;
        const BwdItem e = bwd_item<CAUSAL>(p, item);
        const int kg = e.jb * 128 + r;
        __nv_bfloat16* out = (grp ? p.dv_out : p.dk_out) + ((size_t)e.bh * N + kg) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tAcc + 32 * c, v);
          tmem_wait_ld();
          reg_fence32(v);
          if (kg < N) {
            uint32_t w16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w16[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
            if (p.out_align32) {
              // whole 32-byte sectors (a thread's row is contiguous)
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
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// dQ = scale * dQ_acc, fp32 -> bf16 (round to nearest even), 8 elements per
// thread per step.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    fa_dq_convert_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, float scale,
                         long long n8) {
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n8;
       idx += (long long)gridDim.x * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(dq_acc) + 2 * idx);
    const float4 b = __ldg(reinterpret_cast<const float4*>(dq_acc) + 2 * idx + 1);
    uint4 w;
    w.x = pack_bf16x2(a.x * scale, a.y * scale);
    w.y = pack_bf16x2(a.z * scale, a.w * scale);
    w.z = pack_bf16x2(b.x * scale, b.y * scale);
    w.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[idx] = w;
  }
}

}  // namespace fa
