// Forward kernel: exact softmax attention with the online softmax.
//
// "Interrogating the GPU part 5: FlashAttention", "How does tiling remove the
// traffic?" (a query block stays on chip while key/value blocks stream past)
// and "How can you softmax a row you never see whole?" (running max m,
// running sum l, rescaled accumulator; O = o / l at the end); "LLM Flash
// Attention", "End-to-end flow" (one write of O and of the per-row LSE;
// causal block skipping).  Blackwell form of the parts named in
// "Why did Blackwell need FlashAttention-4?": accumulators in tensor memory,
// conditional rescaling.
//
// The work item is a pair of 128-row query tiles (a "tile pair") of one
// (batch, head).  The kernel is persistent: one CTA per SM walks a fixed
// sequence of items (fwd_item below), and the roles run on from one item to
// the next without draining, so the next pair's queries load while the
// tensor core finishes the current pair and its epilogue overlaps the next
// pair's first score products.  Warp roles (384 threads):
//   warps 0-3  softmax warpgroup of tile 0 (thread = query row)
//   warps 4-7  softmax warpgroup of tile 1
//   warp  8    issues the score products S = Q K^T (one thread); TMEM owner
//   warp  9    TMA producer (one thread)
//   warp  10   issues the output products O += P V (one thread)
//   warp  11   no role: it completes the third warpgroup, whose registers
//              (setmaxnreg) go to the softmax warpgroups
// The MMA queue of an SM is shallow: a thread that waits or keeps books
// between groups of MMAs leaves the tensor core idle, so the two kinds of
// product are issued by two threads whose waits overlap each other's MMAs.
// Tensor memory (512 columns): one score buffer S (128 fp32 columns) that the
// two tiles use in turn (at d = 64 one per tile), the bf16 probabilities
// P_0, P_1 (64 columns each) and the output accumulators O_0, O_1 (d columns
// each).  Shared memory: Q_0, Q_1 and a ring of K/V tiles, all with 128-byte
// swizzle.  The FP8 instance (FwdCfg<D, true>) keeps this structure with
// E4M3 operands; its differences are described at FwdCfg.
//
// Per key block j the tiles alternate on S: S_0(j), S_1(j), S_0(j+1), ...; a
// softmax releases S as soon as it has loaded its scores into registers, so
// each warpgroup exponentiates while the tensor core computes the other
// tile's scores and output products.  Before overwriting P_t and correcting
// O_t a softmax waits until O_t += P_t(j-1) V_{j-1} has completed.
//
// Scores are handled in base 2: the softmax works on s * scale * log2(e), so
// each probability is one ex2; LSE is converted back to natural-log units.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "sm103_ptx.cuh"

namespace fa {

// Conditional rescale threshold (log2 units): the running maximum used as the
// exponent reference is only moved when a block raises the row maximum by
// more than this, so probabilities stay below 2^8 and most blocks skip the
// correction of l and O.  Any value gives the same result in exact
// arithmetic because l, O and the LSE all use the same reference.
constexpr float kRescaleThresholdLog2 = 8.0f;

constexpr uint64_t kDrainLimitNs = 200ull * 1000 * 1000;  // waits while draining after an abort

// 2^x on the FMA pipe, the software exponential of "Interrogating the GPU
// part 5: FlashAttention", "Why did Blackwell need FlashAttention-4?":
// 2^x = 2^n 2^f with n = floor(x), f = x - n in [0, 1), and 2^f taken as the
// cubic 1 + 0.6951 f + 0.2276 f^2 + 0.0771 f^3 (relative error <= 1.0e-4,
// largest as f -> 1; a bf16 probability's rounding is 2^-9).  floor(x) comes
// from adding 1.5 * 2^23 rounded toward -inf, which leaves it as the integer
// in the low mantissa bits; 2^n is applied by adding n to the exponent field.
// x is clamped below at -127: x = -127 (and -inf) gives exactly 0, x in
// (-127, -126) a value below 2^-126 that the flush-to-zero arithmetic
// downstream treats as 0.  Arguments here never exceed the rescale threshold
// (8), far from the upper end of the exponent range.
__device__ __forceinline__ float ex2_cubic(float x) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  x = fmaxf(x, -127.f);
  const float t = __fadd_rd(x, kMagic);
  const float f = x - (t - kMagic);  // both subtractions exact: f = x - floor(x)
  float p = fmaf(f, 0.0771f, 0.2276f);
  p = fmaf(p, f, 0.6951f);
  p = fmaf(p, f, 1.f);
  return __uint_as_float(__float_as_uint(p) + ((__float_as_uint(t) - __float_as_uint(kMagic)) << 23));
}

// FP8: the E4M3 variant of the same kernel (fa_fwd_fp8): Q and K arrive
// rotated and quantised per 128-row block, V quantised per channel and stored
// transposed per key block (d rows of 128 keys, K-major), P is rounded to E4M3
// for the P V product, and the per-block and per-channel scales are applied to
// the scores and to O.
template <int D, bool FP8 = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!FP8 || D == 128, "the FP8 forward is built for d = 128");
  static constexpr int kTileRows = 128;
  static constexpr int kElemBytes = FP8 ? 1 : 2;
  static constexpr int kTileBytes = kTileRows * D * kElemBytes;  // Q, K, V tiles
  static constexpr int kAtoms = D * kElemBytes / 128;             // 128-byte atom columns per tile
  static constexpr int kAtomElems = 128 / kElemBytes;             // elements per atom row
  static constexpr int kKSteps = D * kElemBytes / 32;             // MMAs of the S product (32 bytes of K each)
  static constexpr int kThreads = 384;  // 12 warps: three whole warpgroups (the register split)
  static constexpr int kLaunchRegs = 168;  // 65536 / 384, rounded down to a multiple of 8
  // Register budgets per thread after setmaxnreg: each SM sub-partition holds
  // one warp of every warpgroup, so 2 kSoftRegs + kMiscRegs = 3 x 168 uses
  // exactly the registers the block was launched with (168 per thread, which
  // the host checks before launching).  Measured: 216 for the softmax warps
  // at d = 64 (+7 %) and in FP8, 208 for bf16 at d = 128 (216 lost 1 % there).
  static constexpr uint32_t kSoftRegs = (D == 64 || FP8) ? 216 : 208;
  static constexpr uint32_t kMiscRegs = 3 * kLaunchRegs - 2 * kSoftRegs;
  static_assert(kSoftRegs % 8 == 0 && kSoftRegs <= 256 && kMiscRegs % 8 == 0 && kMiscRegs >= 24,
                "setmaxnreg takes multiples of 8 in [24, 256]");
  static_assert(kSoftRegs > kLaunchRegs && kMiscRegs < kLaunchRegs, "setmaxnreg.inc raises, .dec lowers");
  static constexpr uint32_t kTmemCols = 512;
  // In FP8 the tensor core also forms the row sums of the rounded P that the
  // output product uses: V^T (read K-major) is followed by 16 rows of E4M3
  // ones, the product O += P [V | 1] is 16 columns wider, and those columns
  // hold sum_k P_rk, rescaled together with O.  In bf16 the softmax sums the
  // rounded values itself.
  static constexpr bool kSumByMma = FP8;
  static constexpr int kOCols = kSumByMma ? D + 16 : D;  // O accumulator columns
  static constexpr int kOnesBytes = FP8 ? 16 * 128 : 0;
  // bf16: O is normalised by the fp32 sum plus the rounding error of each key
  // block's largest probability (see the softmax)
  static constexpr bool kBlockMaxCorr = !FP8;
  // bf16 d = 64: the scores come out of TMEM in two halves, and the maximum of
  // the first is taken while the second loads.  (Measured at d = 64 only
  // together with kBlockMaxCorr there: either alone ran slower through the
  // register allocation; at d = 128 it cost 3.6 % at N = 2048.)
  static constexpr bool kSplitLoad = !FP8 && D == 64;
  // bf16 d = 64: a score buffer per tile (S_0 first, S_1 after the O
  // accumulators: 128 + 2 x 64 + 2 x 64 + 128 = 512 columns), so that a tile's
  // next scores never wait for the other tile to load its own.  At d = 128
  // (and in FP8) the two tiles share one buffer and take turns on it.
  static constexpr bool kDualS = !FP8 && (D == 64);
  // K_j is ring fill 2j, V_j fill 2j+1; with the ones tiles the slots come in
  // pairs (K, V, ones), so the slot count is even
  static constexpr int kSlots = FP8 ? 10 : ((D == 128) ? 5 : 12);
  static_assert(!kSumByMma || kSlots % 2 == 0, "K/V slot pairs");
  static constexpr int kStageBytes = 2 * kTileBytes + kOnesBytes;
  static constexpr int kRingBytes = kSumByMma ? (kSlots / 2) * kStageBytes : kSlots * kTileBytes;
  static __device__ __host__ constexpr int slot_offset(int s) {
    return kSumByMma ? (s / 2) * kStageBytes + (s & 1) * kTileBytes : s * kTileBytes;
  }
  // P of one tile: 128 keys, two bf16 or four E4M3 per column
  static constexpr uint32_t kPCols = FP8 ? 32 : 64;
  static constexpr uint32_t kSCol = 0, kPCol0 = 128, kPCol1 = 128 + kPCols;
  static constexpr uint32_t kOCol0 = 128 + 2 * kPCols, kOCol1 = kOCol0 + kOCols;
  static constexpr uint32_t kSCol1 = kDualS ? kOCol1 + kOCols : kSCol;  // tile 1's score buffer
  static_assert(!kDualS || kSCol1 + 128 <= kTmemCols, "tensor memory budget");
  static_assert(kOCol1 + kOCols <= kTmemCols, "tensor memory budget");
  static constexpr int kSmemBytes = 1024 + 2 * kTileBytes + kRingBytes + 512;
};

struct FwdBarriers {
  uint64_t q_full;
  uint64_t q_empty;     // the S products of the CTA's current tile pair are complete (MMA commit)
  uint64_t kv_full[16];
  uint64_t kv_empty[16];
  uint64_t s_full[2];   // S holds tile t's scores (MMA commit)
  uint64_t s_free[2];   // the tile that used a score buffer last has loaded it (128 softmax threads;
                        // one buffer, index 0, unless each tile has its own)
  uint64_t p_full[2];   // P_t written, O_t corrected (128 softmax threads)
  uint64_t pv_done[2];  // O_t += P_t V complete (MMA commit)
  uint64_t drain[2];    // one per issuing thread
  uint64_t never;  // signalled by nothing: the debug stall waits on it
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(FwdBarriers) <= 512, "barriers overflow their shared-memory slot");

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int N;
  int num_pairs;   // tile pairs per (batch, head)
  int num_bh;      // B * H
  int pair_items;  // pairs (by rank) processed as pairs; the rest as single tiles
  int num_items;   // pair_items + 2 (num_pairs num_bh - pair_items)
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  int debug_stall;  // nonzero: the MMA thread first waits on `never` (tests the timeout path)
  int o_align32;    // nonzero: o is 32-byte aligned, so O rows are written in 32-byte stores
  // FP8 only: dequantisation scales
  const float* q_scale;  // [B*H][nkb]: query block scales
  const float* k_scale;  // [B*H][nkb]: key block scales
  const float* v_scale;  // [B*H][D]: value channel scales
  int nkb;               // 128-row blocks per head
};

// wait sites reported in the status word
enum : int { kSiteStall = 0, kSiteFwdProducer = 1, kSiteFwdQ, kSiteFwdK, kSiteFwdV, kSiteFwdSFree, kSiteFwdP,
             kSiteFwdS, kSiteFwdO, kSiteFwdPvDone, kSiteFwdQEmpty };

// One work item: a pair of 128-row query tiles of one (batch, head), or a
// single tile (nb1 = 0).
struct FwdItem {
  int bh;
  int q0;        // first query row of tile 0
  int nb0, nb1;  // key blocks visited by tile 0 and tile 1 (0: no such tile)
};

// The CTAs are persistent: CTA c takes, in round k, the item of rank
// k G + c (even k) or k G + G - 1 - c (odd k), G = gridDim.x.  Pairs are
// ranked so that consecutive ranks cost about the same: with the causal mask
// the cost of a pair grows with its position, and the ranks run over the
// pairs from the last (heaviest) to the first, each pair across all heads;
// the alternating direction then evens out the CTAs' totals.  Without the
// mask every pair costs the same and the ranks run head by head, so that
// the CTAs working at the same time share each head's keys and values in L2.
// The pairs of rank >= pair_items are split into their two tiles, each an
// item of its own (ranks pair_items + 2 (rank - pair_items) + tile), so that
// a last round with fewer pairs than CTAs takes about the time of one tile.
template <bool CAUSAL>
__device__ __forceinline__ bool fwd_item(const FwdParams& p, int k, FwdItem& w) {
  // (ranks fit in int: there are fewer than 2^31 / 2^14 items, see fa_fwd's limits)
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const int r = k * G + ((k & 1) ? G - 1 - c : c);
  if (r >= p.num_items) return false;
  const bool single = r >= p.pair_items;
  const int pr = single ? p.pair_items + ((r - p.pair_items) >> 1) : r;  // pair rank
  int pair;
  if (CAUSAL) {
    pair = p.num_pairs - 1 - pr / p.num_bh;
    w.bh = pr % p.num_bh;
  } else {
    pair = pr % p.num_pairs;
    w.bh = pr / p.num_pairs;
  }
  const int nblk = (p.N + 127) / 128;
  if (single) {
    const int tile = (r - p.pair_items) & 1;
    w.q0 = pair * 256 + 128 * tile;
    w.nb0 = w.q0 < p.N ? (CAUSAL ? min(nblk, 2 * pair + 1 + tile) : nblk) : 0;  // 0: past N, nothing to do
    w.nb1 = 0;
  } else {
    w.q0 = pair * 256;
    w.nb0 = CAUSAL ? min(nblk, 2 * pair + 1) : nblk;
    w.nb1 = w.q0 + 128 < p.N ? (CAUSAL ? min(nblk, 2 * pair + 2) : nblk) : 0;
  }
  return true;
}


// SOFT_EXP: of every four pairs of probabilities a softmax thread forms, the
// first SOFT_EXP pairs take ex2_cubic on the FMA pipe and the rest the MUFU's
// ex2.approx (0: all on the MUFU).
template <int D, bool CAUSAL, bool FP8 = false, int SOFT_EXP = 0>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + 2 * C::kTileBytes;
  FwdBarriers* bar = reinterpret_cast<FwdBarriers*>(sKV + C::kRingBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;

  if (C::kSumByMma) {
    // (FP8) the E4M3 ones (0x38) after each V^T slot, read by the tensor core
    const uint32_t one = 0x38383838u;
    for (int st = 0; st < C::kSlots / 2; ++st) {
      uint4* ones = reinterpret_cast<uint4*>(sKV + st * C::kStageBytes + 2 * C::kTileBytes);
      for (int i = tid; i < C::kOnesBytes / 16; i += C::kThreads) ones[i] = make_uint4(one, one, one, one);
    }
    fence_async_shared();
  }
  if (tid == 0) {
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_empty, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar->kv_full[s], 1);
      mbar_init(&bar->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar->s_full[t], 1);
      mbar_init(&bar->p_full[t], 128);
      mbar_init(&bar->pv_done[t], 1);
    }
    mbar_init(&bar->s_free[0], 128);
    mbar_init(&bar->s_free[1], 128);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtx ctx{&bar->abort_flag, p.wait_limit_ns};

  // Every role walks the same sequence of items; the ring fills, the uses of
  // S and the per-tile products are counted across items, so barrier phases
  // carry over from one item to the next.
  // Register split: the issuing and producer warpgroup (warps 8-11; warp 11
  // has no role and is there to make the warpgroup whole) gives registers
  // back down to C::kMiscRegs a thread, the two softmax warpgroups take
  // C::kSoftRegs.
  if (warp >= 8) {
    setmaxnreg_dec<C::kMiscRegs>();
    if (warp == 9) {
      // ------------------------------------------------------------------ TMA producer
      // fill order = consumption order: K_0, V_0, K_1, V_1, ... of each item in turn
      if (lane == 0) {
        int fill = 0, nq = 0;
        bool ok = true;
        auto load_kv = [&](int j, int kv, int bh) -> bool {
          const int s = fill % C::kSlots;
          const uint32_t u = fill / C::kSlots;
          if (!wait_bounded_inl(&bar->kv_empty[s], (u & 1) ^ 1, ctx, kSiteFwdProducer)) return false;
          mbar_arrive_expect_tx(&bar->kv_full[s], C::kTileBytes);
          if (FP8 && kv) {
            // V^T of key block j: d rows of 128 keys, tile (bh, j) of the transposed layout
            tma_load_3d(sKV + C::slot_offset(s), &map_v, &bar->kv_full[s], 0, 0, bh * p.nkb + j);
          } else {
            const CUtensorMap* map = kv ? &map_v : &map_k;
            for (int a = 0; a < C::kAtoms; ++a)
              tma_load_3d(sKV + C::slot_offset(s) + a * 16384, map, &bar->kv_full[s], a * C::kAtomElems, j * 128, bh);
          }
          ++fill;
          return true;
        };
        FwdItem w;
        for (int k = 0; ok && fwd_item<CAUSAL>(p, k, w); ++k) {
          const int nb_max = max(w.nb0, w.nb1);
          if (nb_max == 0) continue;  // a single tile past N
          const bool has1 = w.nb1 > 0;
          // the first key/value block needs only ring slots: it goes out
          // before Q, whose buffer the previous item may still be reading
          ok = load_kv(0, 0, w.bh) && load_kv(0, 1, w.bh);
          if (ok && nq > 0) ok = wait_bounded_inl(&bar->q_empty, (nq - 1) & 1, ctx, kSiteFwdQEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar->q_full, C::kTileBytes * (has1 ? 2 : 1));
          for (int t = 0; t < (has1 ? 2 : 1); ++t)
            for (int a = 0; a < C::kAtoms; ++a)
              tma_load_3d(sQ + t * C::kTileBytes + a * 16384, &map_q, &bar->q_full, a * C::kAtomElems, w.q0 + 128 * t,
                          w.bh);
          ++nq;
          // the next item's queries go to L2 now, so that their load at the
          // item boundary is served from there
          FwdItem nx;
          if (fwd_item<CAUSAL>(p, k + 1, nx) && nx.nb0 > 0)
            for (int t = 0; t < (nx.nb1 > 0 ? 2 : 1); ++t)
              for (int a = 0; a < C::kAtoms; ++a)
                tma_prefetch_l2_3d(&map_q, a * C::kAtomElems, nx.q0 + 128 * t, nx.bh);
          for (int j = 1; ok && j < nb_max; ++j) ok = load_kv(j, 0, w.bh) && load_kv(j, 1, w.bh);
        }
        // every copy this thread started must land before the CTA can exit
        if (nq > 0) wait_drain_inl(&bar->q_full, (nq - 1) & 1, kDrainLimitNs);
        for (int s = 0; s < C::kSlots; ++s) {
          if (fill > s) {
            const int uses = (fill - 1 - s) / C::kSlots + 1;
            wait_drain_inl(&bar->kv_full[s], (uses - 1) & 1, kDrainLimitNs);
          }
        }
      }
      __syncwarp();
    } else if (warp == 8) {
      // ------------------------------------------------------------------ S issuer
      // K_j is ring fill 2g (g counts key blocks over all items); S(k) waits
      // until the tile that used S before has loaded it
      if (lane == 0) {
        const uint32_t sq = smem_u32(sQ), skv = smem_u32(sKV);
        const uint64_t qdesc0 = sdesc_sw128(sq, 16, 1024);
        const uint64_t qdesc1 = sdesc_sw128(sq + C::kTileBytes, 16, 1024);
        constexpr uint32_t id_s = FP8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
        int s_uses[2] = {0, 0}, g = 0, nq = 0;  // S products issued into each score buffer
        bool ok = !(p.debug_stall && !wait_bounded_inl(&bar->never, 0, ctx, kSiteStall));
        FwdItem w;
        for (int k = 0; ok && fwd_item<CAUSAL>(p, k, w); ++k) {
          const int nb_max = max(w.nb0, w.nb1);
          if (nb_max == 0) continue;
          if (!wait_bounded_inl(&bar->q_full, nq & 1, ctx, kSiteFwdQ)) break;
          ++nq;
          for (int j = 0; ok && j < nb_max; ++j, ++g) {
            const int f = 2 * g;
            const int ks = f % C::kSlots;
            if (!wait_bounded_inl(&bar->kv_full[ks], (f / C::kSlots) & 1, ctx, kSiteFwdK)) {
              ok = false;
              break;
            }
            const uint64_t kdesc = sdesc_sw128(skv + C::slot_offset(ks), 16, 1024);
  #pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (j < (t ? w.nb1 : w.nb0)) {
                const int sb = C::kDualS ? t : 0;
                if (s_uses[sb] > 0 && !wait_bounded_inl(&bar->s_free[sb], (s_uses[sb] - 1) & 1, ctx, kSiteFwdSFree)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t qd = t ? qdesc1 : qdesc0;
  #pragma unroll
                for (int kk = 0; kk < C::kKSteps; ++kk) {
                  const uint32_t off = (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                  const uint32_t scol = tmem + (sb ? C::kSCol1 : C::kSCol);
                  if constexpr (FP8)
                    mma_e4m3_ss(scol, qd + off, kdesc + off, id_s, kk > 0 ? 1u : 0u);
                  else
                    mma_bf16_ss(scol, qd + off, kdesc + off, id_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar->s_full[t]);
                ++s_uses[sb];
              }
            }
            if (!ok) break;
            mma_commit(&bar->kv_empty[ks]);
          }
          if (!ok) break;
          // the item's queries have been read: their buffer may take the next item's
          mma_commit(&bar->q_empty);
        }
        // everything issued must complete before the tensor memory is released
        mma_commit(&bar->drain[0]);
        wait_drain_inl(&bar->drain[0], 0, kDrainLimitNs);
      }
      __syncwarp();
    } else if (warp == 10) {
      // ------------------------------------------------------------------ P V issuer
      // V_j is ring fill 2g+1; O_t += P_t(j) V_j once the softmax of tile t wrote P_t(j)
      if (lane == 0) {
        const uint32_t skv = smem_u32(sKV);
        // bf16: V read N-major; FP8: V^T read K-major (with the ones rows after it)
        constexpr uint32_t id_pv = FP8 ? idesc_e4m3_f32(128, C::kOCols) : idesc_bf16_f32(128, C::kOCols, false, true);
        int g = 0;
        int pv_uses[2] = {0, 0};
        bool ok = true;
        FwdItem w;
        for (int k = 0; ok && fwd_item<CAUSAL>(p, k, w); ++k) {
          const int nb_max = max(w.nb0, w.nb1);
          if (nb_max == 0) continue;
          for (int j = 0; ok && j < nb_max; ++j, ++g) {
            const int f = 2 * g + 1;
            const int vs = f % C::kSlots;
            if (!wait_bounded_inl(&bar->kv_full[vs], (f / C::kSlots) & 1, ctx, kSiteFwdV)) {
              ok = false;
              break;
            }
            // (FP8: the ones rows after V^T make the last 16 columns of O the row sums)
            const uint64_t vdesc = sdesc_sw128(skv + C::slot_offset(vs), FP8 ? 16 : 16384, 1024);
  #pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (j < (t ? w.nb1 : w.nb0)) {
                if (!wait_bounded_inl(&bar->p_full[t], pv_uses[t] & 1, ctx, kSiteFwdP)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint32_t dcol = tmem + (t ? C::kOCol1 : C::kOCol0);
                const uint32_t pcol = tmem + (t ? C::kPCol1 : C::kPCol0);
                if constexpr (FP8) {
                  // 4 steps of 32 keys: P from 8 TMEM columns each, V^T rows at +32 bytes
  #pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    mma_e4m3_ts(dcol, pcol + kk * 8, vdesc + (uint32_t)((kk * 32) >> 4), id_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                } else {
  #pragma unroll
                  for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(dcol, pcol + kk * 8, vdesc + (uint32_t)((kk * 2048) >> 4), id_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bar->pv_done[t]);
                ++pv_uses[t];
              }
            }
            if (!ok) break;
            mma_commit(&bar->kv_empty[vs]);
          }
        }
        mma_commit(&bar->drain[1]);
        wait_drain_inl(&bar->drain[1], 0, kDrainLimitNs);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<C::kSoftRegs>();
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + ((C::kDualS && t) ? C::kSCol1 : C::kSCol) + lane_off;
    const uint32_t tP = tmem + (t ? C::kPCol1 : C::kPCol0) + lane_off;
    const uint32_t tO = tmem + (t ? C::kOCol1 : C::kOCol0) + lane_off;
    const float sl2 = p.scale_log2;
    int uses = 0;  // blocks this tile has processed over all items (= S loads = P V products)
    bool alive = true;
    FwdItem w;
    for (int k = 0; alive && fwd_item<CAUSAL>(p, k, w); ++k) {
      const int nb = t ? w.nb1 : w.nb0;
      if (nb == 0) continue;
      const int row_q0 = w.q0 + 128 * t;  // first query row of this tile
      const int row_g = row_q0 + r;
      // FP8: the scores are the E4M3 products times the query and key block scales
      const float qsl2 = FP8 ? sl2 * __ldg(p.q_scale + (size_t)w.bh * p.nkb + (row_q0 >> 7)) : sl2;
      float m = -CUDART_INF_F;  // exponent reference (log2 units), a stale running max
      // l: sum of the fp32 probabilities (for the LSE); lcorr (bf16): the
      // rounding errors of each key block's largest probability, so that
      // l + lcorr normalises O (below); l_mma: the normaliser (FP8: the sum of
      // the rounded probabilities, formed by the tensor core)
      float l = 0.f, lcorr = 0.f, l_mma = 0.f;
      for (int j = 0; j < nb; ++j, ++uses) {
        // score factor of this key block (loaded before the wait hides its latency)
        const float cj = FP8 ? qsl2 * __ldg(p.k_scale + (size_t)w.bh * p.nkb + j) : sl2;
        if (!__all_sync(0xffffffffu, wait_bounded_inl(&bar->s_full[t], uses & 1, ctx, kSiteFwdS))) {
          alive = false;
          break;
        }
        tc_fence_after();
        // the maximum of 64 scores: a tree of 3-input maxima
        auto max64 = [](const uint32_t* x, const uint32_t* y) {
          float t1[22];
#pragma unroll
          for (int i = 0; i < 21; ++i) {
            const int e = 3 * i;
            t1[i] = max3(__uint_as_float(e < 32 ? x[e] : y[e - 32]), __uint_as_float(e + 1 < 32 ? x[e + 1] : y[e - 31]),
                         __uint_as_float(e + 2 < 32 ? x[e + 2] : y[e - 30]));
          }
          t1[21] = __uint_as_float(y[31]);
          float t2[8];
#pragma unroll
          for (int i = 0; i < 7; ++i) t2[i] = max3(t1[3 * i], t1[3 * i + 1], t1[3 * i + 2]);
          t2[7] = t1[21];
          return max3(max3(t2[0], t2[1], t2[2]), max3(t2[3], t2[4], t2[5]), fmaxf(t2[6], t2[7]));
        };
        uint32_t sr[4][32];
        float mx_a = 0.f;  // kSplitLoad: the maximum of the first 64 scores, unmasked
        if constexpr (C::kSplitLoad) {
          tmem_ld32(tS, sr[0]);
          tmem_ld32(tS + 32, sr[1]);
          tmem_wait_ld();
          reg_fence32(sr[0]);
          reg_fence32(sr[1]);
          tmem_ld32(tS + 64, sr[2]);
          tmem_ld32(tS + 96, sr[3]);
          mx_a = max64(sr[0], sr[1]);
          tmem_wait_ld();
          reg_fence32(sr[2]);
          reg_fence32(sr[3]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sr[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) reg_fence32(sr[c]);
        }
        // the scores are in registers: the next scores may now overwrite S
        tc_fence_before();
        mbar_arrive(&bar->s_free[C::kDualS ? t : 0]);

        const int kbase = j * 128;
        const bool tail = kbase + 128 > N;
        const bool diag = CAUSAL && (kbase + 127 > row_q0);
        if (tail || diag) {
          const int last = (CAUSAL ? min(N - 1, row_g) : N - 1) - kbase;  // last visible key of this row
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > last) sr[c >> 5][c & 31] = __float_as_uint(-CUDART_INF_F);
        }
        // row maximum as a tree of 3-input maxima (kSplitLoad: the two
        // halves'; a masked block takes the first half again)
        float mx;
        if constexpr (C::kSplitLoad) {
          mx = fmaxf((tail || diag) ? max64(sr[0], sr[1]) : mx_a, max64(sr[2], sr[3]));
        } else {
          float t1[43];
#pragma unroll
          for (int i = 0; i < 42; ++i)
            t1[i] = max3(__uint_as_float(sr[(3 * i) >> 5][(3 * i) & 31]),
                         __uint_as_float(sr[(3 * i + 1) >> 5][(3 * i + 1) & 31]),
                         __uint_as_float(sr[(3 * i + 2) >> 5][(3 * i + 2) & 31]));
          t1[42] = fmaxf(__uint_as_float(sr[3][30]), __uint_as_float(sr[3][31]));
          float t2[15];
#pragma unroll
          for (int i = 0; i < 14; ++i) t2[i] = max3(t1[3 * i], t1[3 * i + 1], t1[3 * i + 2]);
          t2[14] = t1[42];
          float t3[5];
#pragma unroll
          for (int i = 0; i < 5; ++i) t3[i] = max3(t2[3 * i], t2[3 * i + 1], t2[3 * i + 2]);
          mx = max3(max3(t3[0], t3[1], t3[2]), t3[3], t3[4]);
        }
        const float m_new = fmaxf(m, mx * cj);
        // conditional rescale: move the exponent reference only when the row
        // maximum rose by more than the threshold (always on the first block)
        float alpha = 1.f;
        bool rescale_warp = false;
        if (j == 0) {
          m = m_new;
        } else {
          const bool need = (m_new - m) > kRescaleThresholdLog2;
          rescale_warp = __any_sync(0xffffffffu, need);
          if (need) {
            alpha = ex2_approx(m - m_new);
            m = m_new;
          }
        }
        // p = 2^(s c - m) two at a time, with their fp32 sum (four partial sums).
        const float2 c2 = make_float2(cj, cj);
        const float2 mneg2 = make_float2(-m, -m);
        float2 acc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = make_float2(0.f, 0.f);
        if (C::kBlockMaxCorr) {
          // The P V product uses bf16-rounded probabilities.  O is normalised
          // by l plus the rounding error of each block's largest probability:
          // a dominant probability (up to 2^8 with the stale reference) then
          // cancels exactly between numerator and normaliser, as it would with
          // the sum of all the rounded values, and the block's smaller
          // probabilities leave only their small, random rounding errors.  The
          // block maximum's exponent argument is the same fused multiply-add
          // the loop below forms for it, so the value is bit-identical.
          const float pbm = ex2_approx(fmaf(mx, cj, -m));
          const float pbm_r = __uint_as_float(pack_bf16x2(pbm, 0.f) << 16);
          lcorr = lcorr * alpha + (pbm_r - pbm);
        }
        // (in FP8 the sums of the rounded values come from the tensor core)
        // bf16: two probabilities per 32-bit word; FP8: four (pk[c][0..7] used)
        uint32_t pk[4][16];
        float hold0 = 0.f, hold1 = 0.f;  // (FP8) the previous pair until its word of four is complete
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])),
                                        c2, mneg2);
            float p0, p1;
            if (SOFT_EXP > 0 && (i & 3) < SOFT_EXP) {
              p0 = ex2_cubic(x.x);
              p1 = ex2_cubic(x.y);
            } else {
              p0 = ex2_approx(x.x);
              p1 = ex2_approx(x.y);
            }
            if constexpr (FP8) {
              if (i & 1) {
                pk[c][i >> 1] = pack_e4m3x4(hold0, hold1, p0, p1);
              } else {
                hold0 = p0;
                hold1 = p1;
              }
            } else {
              pk[c][i] = pack_bf16x2(p0, p1);
            }
            acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
          }
        }
        const float2 accs = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        l = l * alpha + (accs.x + accs.y);
        // P_t and O_t are in use until O_t += P_t(j-1) V_{j-1} has completed
        // (at j = 0 the previous item's epilogue has already waited for its
        // last product)
        if (j > 0) {
          if (!__all_sync(0xffffffffu, wait_bounded_inl(&bar->pv_done[t], (uses - 1) & 1, ctx, kSiteFwdPvDone))) {
            alive = false;
            break;
          }
          tc_fence_after();
        }
        if (rescale_warp) {
          // correction O <- alpha O, in place in tensor memory
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + 32 * c, ov);
            tmem_wait_ld();
            reg_fence32(ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tO + 32 * c, ov);
          }
          if (C::kSumByMma) {
            // the row sums of the rounded P are rescaled with O
            uint32_t sv[16];
            tmem_ld16(tO + D, sv);
            tmem_wait_ld();
            reg_fence16(sv);
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[i] = __float_as_uint(__uint_as_float(sv[i]) * alpha);
            tmem_st16(tO + D, sv);
          }
          tmem_wait_st();
        }
        if constexpr (FP8) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_st8(tP + 8 * c, pk[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_st16(tP + 16 * c, pk[c]);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar->p_full[t]);
      }
      if (!alive) break;
      // epilogue: O = o / l_mma (in FP8 from the extra O columns), LSE = (m + log2 l) ln 2.
      // Once the tensor memory loads below have completed, the next item's
      // first P V product may overwrite O_t (it is issued only after this
      // warpgroup has written the next P_t).
      if (!__all_sync(0xffffffffu, wait_bounded_inl(&bar->pv_done[t], (uses - 1) & 1, ctx, kSiteFwdO))) {
        alive = false;
        break;
      }
      tc_fence_after();
      if (C::kSumByMma) {
        uint32_t sv[16];
        tmem_ld16(tO + D, sv);
        tmem_wait_ld();
        reg_fence16(sv);
        l_mma = __uint_as_float(sv[0]);
      }
      if (C::kBlockMaxCorr) l_mma = l + lcorr;
      const float inv_l = 1.f / l_mma;
      fwd_item<CAUSAL>(p, k, w);  // (recomputed rather than kept live through the loop)
      __nv_bfloat16* orow = p.o + ((size_t)w.bh * N + row_g) * D;
      // all of O_t's columns in one round trip to tensor memory (four
      // dependent round trips cost ~2.5-3.5k cycles at each item's end)
      uint32_t ovall[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + 32 * c, ovall[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) reg_fence32(ovall[c]);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t* ov = ovall[c];
        if constexpr (FP8) {
          // the value channel scales (the same for every row: broadcast loads)
          const float4* vs4 = reinterpret_cast<const float4*>(p.v_scale + (size_t)w.bh * D + 32 * c);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 sv = __ldg(vs4 + q4);
            ov[4 * q4 + 0] = __float_as_uint(__uint_as_float(ov[4 * q4 + 0]) * sv.x);
            ov[4 * q4 + 1] = __float_as_uint(__uint_as_float(ov[4 * q4 + 1]) * sv.y);
            ov[4 * q4 + 2] = __float_as_uint(__uint_as_float(ov[4 * q4 + 2]) * sv.z);
            ov[4 * q4 + 3] = __float_as_uint(__uint_as_float(ov[4 * q4 + 3]) * sv.w);
          }
        }
        if (row_g < N) {
          uint32_t w16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w16[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
          if (p.o_align32) {
            // whole 32-byte sectors (a thread's row is contiguous)
            st_global_v8(orow + 32 * c, w16);
            st_global_v8(orow + 32 * c + 16, w16 + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(w16[4 * v4], w16[4 * v4 + 1], w16[4 * v4 + 2], w16[4 * v4 + 3]);
          }
        }
      }
      if (row_g < N) p.lse[(size_t)w.bh * N + row_g] = (m + log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
