// Operand preparation of the FP8 forward (fa_fwd_fp8).
//
// "Interrogating the GPU part 5: FlashAttention", "What did FlashAttention-3
// do with Hopper?": FP8 attention quantises per block after a random
// Hadamard rotation, which spreads outliers across the block; "FlashAttention
// versions", "FlashAttention-3 (2024)": block-level quantisation rather than
// one per-tensor scale.
//
// * Q and K: every row x (d = 128) becomes x R with R = diag(s) H / sqrt(d),
//   H the Sylvester Hadamard matrix and s the caller's random signs; since
//   both are rotated by the same orthogonal R, the scores are unchanged.  Each
//   block of 128 rows of one (batch, head) is then scaled by 448 / max|x R|
//   and rounded to E4M3 (nearest even, saturating); the block's scale
//   max|x R| / 448 is kept for the dequantisation of the scores.
// * V: one scale per channel of one (batch, head) over the whole sequence
//   (max_n |v_nc| / 448), constant along the P V sum, so that it applies once
//   to O.  V is written transposed per key block (d rows of 128 keys, keys
//   past N as zeros), the K-major layout the P V product reads.
#pragma once

#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr float kE4m3Max = 448.f;

// The preparation kernel: persistent CTAs of 128 threads, three per SM.  A
// work item is one 128-row block of one operand of one (batch, head), item
// op (B H nblk) + bh nblk + blk with op 0 = Q, 1 = K, 2 = V; CTA c takes items
// c, c + G, c + 2 G, ... (G = the grid), so that V comes last and is still in
// L2 for its second pass.  Every block arrives by TMA (two boxes
// of 64 channels x 128 rows, 128-byte swizzle, rows past N as zeros) into one
// of two shared-memory buffers: the next item's block loads while the current
// one is converted.  The E4M3 rows of a Q or K block go back into the buffer
// they came from and leave by one TMA store (rows past N are not written).
constexpr int kFp8PrepThreads = 128;
constexpr int kFp8PrepCtasPerSm = 3;
constexpr int kFp8PrepBufBytes = 128 * 256;  // one block, bf16
constexpr int kFp8PrepSmemBytes = 1024 + 2 * kFp8PrepBufBytes + 8 * 128 * 4 + 128 * 4 + 4 * 4 + 4 * 8;
constexpr uint64_t kFp8DrainLimitNs = 200ull * 1000 * 1000;  // waits while draining after an abort
enum : int { kSiteFp8Prep = 64 };

// byte offset of channels 8 g .. 8 g + 7 of row r in a staged block (g < 16)
__device__ __forceinline__ uint32_t fp8_stage_offset(int r, int g) {
  return (uint32_t)((g >> 3) * 16384 + r * 128 + (((g & 7) ^ (r & 7)) << 4));
}

// V, pass 1: per-channel maximum of |v| over one staged key block, folded
// into amax_bits[bh][c] (non-negative floats order like their bit patterns).
// Thread t reads channels 8 (t % 16) .. +7 of rows t / 16, t / 16 + 8, ...
// (a quarter warp covers one row's 128 bytes of a half: no bank conflicts),
// then the 8 row groups are combined through shared memory.  Zero rows past
// N do not change a maximum of absolute values.
__device__ __forceinline__ void fp8_v_amax_block(const uint8_t* stage, unsigned* __restrict__ amax_bits, int bh,
                                                 float (*part)[128]) {
  constexpr int D = 128;
  const int t = threadIdx.x, cg = t & 15, rg = t >> 4;
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = rg + 8 * i;
    const uint4 raw = *reinterpret_cast<const uint4*>(stage + fp8_stage_offset(r, cg));
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      m[2 * e] = fmaxf(m[2 * e], fabsf(f.x));
      m[2 * e + 1] = fmaxf(m[2 * e + 1], fabsf(f.y));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[rg][8 * cg + i] = m[i];
  __syncthreads();
  float mx = part[0][t];
#pragma unroll
  for (int g = 1; g < 8; ++g) mx = fmaxf(mx, part[g][t]);
  atomicMax(amax_bits + (size_t)bh * D + t, __float_as_uint(mx));
}

// bf16 pair (one 32-bit word) -> fp32 with the signs of the rotation applied:
// neg_lo / neg_hi are 0x80000000 to negate that element, else 0.  The low
// element moves to the top half (w * 2^16, plus the sign bit mod 2^32); the
// high element keeps the top half (its sign bit exclusive-or'ed).
__device__ __forceinline__ float2 bf16x2_signed(uint32_t w, uint32_t neg_lo, uint32_t neg_hi) {
  return make_float2(__uint_as_float((w << 16) + neg_lo), __uint_as_float((w & 0xffff0000u) ^ neg_hi));
}

// Q or K block (staged): thread = row; writes the block's E4M3 codes over the
// staged block (the same 128-byte swizzle, 128 bytes a row) for a TMA store.  The row's 128 channels stay in
// registers as 64 pairs y[k] = (x_k, x_{k+64}), and the rotation is a fast
// Walsh-Hadamard transform of the row: butterflies (a, b) -> (a + b, a - b)
// on each bit of the channel index, lowest first: bits 0..5 between pairs,
// two butterflies per packed fp32x2 add and subtract (the subtraction as a
// fused multiply-add by -1: the same value), bit 6 inside each pair.  Then
// the block maximum of |x R| gives the scale, and each thread rounds its row
// to E4M3.
__device__ __forceinline__ void fp8_qk_block(uint8_t* stage, const uint32_t* neg, float* __restrict__ scales, int nblk,
                                             int blk, int bh, float* red) {
  constexpr int kWarps = kFp8PrepThreads / 32;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  float2 y[64];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    // channels 8 c .. 8 c + 7 and 64 + 8 c .. 64 + 8 c + 7
    const uint4 rl = *reinterpret_cast<const uint4*>(stage + fp8_stage_offset(t, c));
    const uint4 rh = *reinterpret_cast<const uint4*>(stage + fp8_stage_offset(t, c + 8));
    const uint32_t wl[4] = {rl.x, rl.y, rl.z, rl.w};
    const uint32_t wh[4] = {rh.x, rh.y, rh.z, rh.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 nl = *reinterpret_cast<const uint4*>(neg + 8 * c + 4 * h);
      const uint4 nh = *reinterpret_cast<const uint4*>(neg + 64 + 8 * c + 4 * h);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int e = 4 * h + 2 * q;  // channels 8 c + e, 8 c + e + 1 (word e / 2)
        const float2 lo = bf16x2_signed(wl[e / 2], q ? nl.z : nl.x, q ? nl.w : nl.y);
        const float2 hi = bf16x2_signed(wh[e / 2], q ? nh.z : nh.x, q ? nh.w : nh.y);
        y[8 * c + e] = make_float2(lo.x, hi.x);
        y[8 * c + e + 1] = make_float2(lo.y, hi.y);
      }
    }
  }
  const float2 minus1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      if (k & h) continue;
      const float2 a = y[k], b = y[k + h];
      y[k] = __fadd2_rn(a, b);
      y[k + h] = __ffma2_rn(b, minus1, a);
    }
  }
  // bit 6, then the 1 / sqrt(d) of R: y[k] = (rotated channel k, channel k + 64)
  const float inv_sqrt_d = 0.08838834764831845f;  // 1 / sqrt(128)
  const float2 isd2 = make_float2(inv_sqrt_d, inv_sqrt_d);
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 64; ++k) {
    const float a = y[k].x, b = y[k].y;
    y[k] = __fmul2_rn(make_float2(a + b, a - b), isd2);
    amax = fmaxf(amax, fmaxf(fabsf(y[k].x), fabsf(y[k].y)));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? amax / kE4m3Max : 1.f;
  const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
  // (every thread has read its row: the block maximum's barrier is behind it)
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    w[j] = pack_e4m3x4(y[4 * j].x * inv, y[4 * j + 1].x * inv, y[4 * j + 2].x * inv, y[4 * j + 3].x * inv);
    w[16 + j] = pack_e4m3x4(y[4 * j].y * inv, y[4 * j + 1].y * inv, y[4 * j + 2].y * inv, y[4 * j + 3].y * inv);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(stage + t * 128 + ((j ^ (t & 7)) << 4)) =
        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_async_shared();
  if (t == 0) scales[(size_t)bh * nblk + blk] = scale;
}

// One launch prepares Q, K (rotation and block quantisation) and the first
// pass over V (channel maxima).
__global__ void __launch_bounds__(kFp8PrepThreads, kFp8PrepCtasPerSm)
    fa_fp8_prepare_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                          const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_q8,
                          const __grid_constant__ CUtensorMap map_k8, const int8_t* __restrict__ signs, float* __restrict__ scales0,
                          float* __restrict__ scales1, unsigned* __restrict__ v_amax_bits, int N, int nblk, int BH,
                          uint64_t wait_limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float(*part)[128] = reinterpret_cast<float(*)[128]>(buf + 2 * kFp8PrepBufBytes);
  uint32_t* neg = reinterpret_cast<uint32_t*>(buf + 2 * kFp8PrepBufBytes + 8 * 128 * 4);  // 0x80000000 where s = -1
  float* red = reinterpret_cast<float*>(neg + 128);
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 4);  // [0], [1]: the two buffers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 2);
  const long long per_op = (long long)BH * nblk, items = 3 * per_op;
  auto load = [&](long long item, int b) {
    const int op = item >= 2 * per_op ? 2 : (item >= per_op ? 1 : 0);
    const long long bb = item - op * per_op;
    const int blk = (int)(bb % nblk), bh = (int)(bb / nblk);
    const CUtensorMap* map = op == 0 ? &map_q : (op == 1 ? &map_k : &map_v);
    mbar_arrive_expect_tx(&bar[b], kFp8PrepBufBytes);  // the whole box, zero rows included
    tma_load_3d(buf + b * kFp8PrepBufBytes, map, &bar[b], 0, blk * 128, bh);
    tma_load_3d(buf + b * kFp8PrepBufBytes + 16384, map, &bar[b], 64, blk * 128, bh);
  };
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (blockIdx.x < items) load(blockIdx.x, 0);
  }
  neg[threadIdx.x] = signs[threadIdx.x] < 0 ? 0x80000000u : 0u;
  __syncthreads();
  const WaitCtx ctx{abort_flag, wait_limit_ns};
  int k = 0;
  for (long long item = blockIdx.x; item < items; item += gridDim.x, ++k) {
    // the next item's block into the other buffer, which the previous
    // iteration has finished with (its barriers), once the TMA store from it
    // has read it
    if (threadIdx.x == 0 && item + gridDim.x < items) {
      bulk_wait_read<0>();
      load(item + gridDim.x, (k + 1) & 1);
    }
    const bool ok = wait_bounded(&bar[k & 1], (k >> 1) & 1, ctx, kSiteFp8Prep);
    if (!__syncthreads_and(ok)) break;
    const int op = item >= 2 * per_op ? 2 : (item >= per_op ? 1 : 0);
    const long long bb = item - op * per_op;
    const int blk = (int)(bb % nblk), bh = (int)(bb / nblk);
    uint8_t* stage = buf + (k & 1) * kFp8PrepBufBytes;
    if (op == 2) {
      fp8_v_amax_block(stage, v_amax_bits, bh, part);
    } else {
      fp8_qk_block(stage, neg, op ? scales1 : scales0, nblk, blk, bh, red);
      __syncthreads();
      if (threadIdx.x == 0) {
        tma_store_3d(op ? &map_k8 : &map_q8, stage, 0, blk * 128, bh);
        tma_store_commit();
      }
    }
    // (the next iteration's first barrier orders this one's reads of the
    // buffer, part and red before anything overwrites them)
  }
  if (threadIdx.x == 0) tma_store_wait_all();
  // after a timeout, the copies in flight land before the CTA ends
  if (threadIdx.x == 0 && *abort_flag) {
    // iteration k stopped: the loads of this CTA's items 0 .. k + 1 (as far as it has items) started
    const long long mine = (items - 1 - blockIdx.x) / gridDim.x + 1;
    const int issued = (int)(k + 2 < mine ? k + 2 : mine);
    for (int b = 0; b < 2; ++b) {
      const int uses = issued > b ? (issued - 1 - b) / 2 + 1 : 0;  // loads into buffer b
      if (uses > 0) wait_drain(&bar[b], (uses - 1) & 1, kFp8DrainLimitNs);
    }
  }
}

// V, pass 2: quantise one key block per channel and write it transposed,
// v8t[bh][blk][c][key] (keys past N as zeros); the blk = 0 CTA also writes
// the channel scales.  256 threads: thread t converts channels 8 (t % 16)
// .. +7 of four consecutive keys at a time (16-byte loads), packs each
// channel's four keys into one word of a shared [channel][key / 4] tile, and
// the tile leaves as 128-byte rows (16-byte stores, consecutive threads on
// consecutive addresses).
__global__ void __launch_bounds__(256)
    fa_fp8_v_quant_kernel(const __nv_bfloat16* __restrict__ v, const unsigned* __restrict__ amax_bits,
                          uint8_t* __restrict__ v8t, float* __restrict__ v_scale, int N, int nblk) {
  constexpr int D = 128, kPad = 33;  // words per tile row: 32 + 1 against bank conflicts
  __shared__ uint32_t tile[D * kPad];
  const int t = threadIdx.x, cg = t & 15, kg = t >> 4, blk = blockIdx.x, bh = blockIdx.y;
  float inv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float amax = __uint_as_float(amax_bits[(size_t)bh * D + 8 * cg + i]);
    inv[i] = amax > 0.f ? kE4m3Max / amax : 1.f;
  }
  const __nv_bfloat16* src = v + ((size_t)bh * N + blk * 128) * D + 8 * cg;
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int kw = kg + 16 * it;  // word of four keys 4 kw .. 4 kw + 3
    float f[4][8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = blk * 128 + 4 * kw + e;
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (key < N) raw = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(4 * kw + e) * D));
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(h2[i]);
        f[e][2 * i] = x.x * inv[2 * i];
        f[e][2 * i + 1] = x.y * inv[2 * i + 1];
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) tile[(8 * cg + i) * kPad + kw] = pack_e4m3x4(f[0][i], f[1][i], f[2][i], f[3][i]);
  }
  __syncthreads();
  uint8_t* dst = v8t + ((size_t)bh * nblk + blk) * D * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int id = t + 256 * i;  // 16-byte chunk id: row id / 8, chunk id % 8
    const int c = id >> 3, q = id & 7;
    const uint32_t* w = tile + c * kPad + 4 * q;
    *reinterpret_cast<uint4*>(dst + (size_t)c * 128 + 16 * q) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (blk == 0 && t < D) {
    const float amax = __uint_as_float(amax_bits[(size_t)bh * D + t]);
    v_scale[(size_t)bh * D + t] = amax > 0.f ? amax / kE4m3Max : 1.f;
  }
}

}  // namespace fa
