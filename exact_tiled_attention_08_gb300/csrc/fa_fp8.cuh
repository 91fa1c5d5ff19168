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

// V, pass 1: per-channel maximum of |v| over one key block, folded into
// amax_bits[bh][c] (non-negative floats order like their bit patterns).
// 512 threads: thread t reads channels 8 (t % 16) .. +7 of rows t / 16,
// t / 16 + 32, ... with 16-byte loads (16 threads per 256-byte row), then the
// 32 row groups are combined through shared memory.
__device__ __forceinline__ void fp8_v_amax_block(const __nv_bfloat16* __restrict__ v, unsigned* __restrict__ amax_bits,
                                                 int N, int blk, int bh, float (*part)[128]) {
  constexpr int D = 128;
  const int t = threadIdx.x, cg = t & 15, rg = t >> 4;
  const int rows = min(128, N - blk * 128);
  const __nv_bfloat16* src = v + ((size_t)bh * N + blk * 128) * D + 8 * cg;
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = rg + 32 * i;
    if (r < rows) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + (size_t)r * D));
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h2[e]);
        m[2 * e] = fmaxf(m[2 * e], fabsf(f.x));
        m[2 * e + 1] = fmaxf(m[2 * e + 1], fabsf(f.y));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[rg][8 * cg + i] = m[i];
  __syncthreads();
  if (t < D) {
    float mx = part[0][t];
#pragma unroll
    for (int g = 1; g < 32; ++g) mx = fmaxf(mx, part[g][t]);
    atomicMax(amax_bits + (size_t)bh * D + t, __float_as_uint(mx));
  }
}

// One launch prepares Q, K (rotation and block quantisation) and the first
// pass over V (channel maxima), one 128-row block of one (batch, head) per
// CTA; blockIdx.z selects the operand: 0 = Q, 1 = K, 2 = V.
//
// Q or K: 512 threads = 16 warps x 8 rows; a row is 32 lanes x 4 consecutive
// channels.  The rotation is a fast Walsh-Hadamard transform: butterflies
// (a, b) -> (a + b, a - b) at strides 1 and 2 inside a lane, 4 ... 64 across
// lanes.
__global__ void __launch_bounds__(512)
    fa_fp8_prepare_kernel(const __nv_bfloat16* __restrict__ x0, const __nv_bfloat16* __restrict__ x1,
                          const __nv_bfloat16* __restrict__ v, const int8_t* __restrict__ signs,
                          uint8_t* __restrict__ x8_0, uint8_t* __restrict__ x8_1, float* __restrict__ scales0,
                          float* __restrict__ scales1, unsigned* __restrict__ v_amax_bits, int N, int nblk) {
  constexpr int D = 128, E = 4, kRows = 8, kWarps = 16;
  __shared__ float red[kWarps];
  __shared__ float part[32][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x, bh = blockIdx.y;
  if (blockIdx.z == 2) {
    fp8_v_amax_block(v, v_amax_bits, N, blk, bh, part);
    return;
  }
  const __nv_bfloat16* x = blockIdx.z ? x1 : x0;
  uint8_t* x8 = blockIdx.z ? x8_1 : x8_0;
  float* scales = blockIdx.z ? scales1 : scales0;
  float sgn[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sgn[e] = (float)signs[lane * E + e];
  const float inv_sqrt_d = 0.08838834764831845f;  // 1 / sqrt(128)
  float xr[kRows][E];
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int row = blk * 128 + warp * kRows + r;
    float a[E] = {0.f, 0.f, 0.f, 0.f};
    if (row < N) {
      const uint2 raw = *reinterpret_cast<const uint2*>(x + ((size_t)bh * N + row) * D + lane * E);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      a[0] = lo.x * sgn[0];
      a[1] = lo.y * sgn[1];
      a[2] = hi.x * sgn[2];
      a[3] = hi.y * sgn[3];
    }
    // strides 1 and 2 (inside the lane)
    float b0 = a[0] + a[1], b1 = a[0] - a[1], b2 = a[2] + a[3], b3 = a[2] - a[3];
    a[0] = b0 + b2;
    a[2] = b0 - b2;
    a[1] = b1 + b3;
    a[3] = b1 - b3;
    // strides 4 .. 64: the partner element sits in lane ^ (stride / 4); the
    // lower element becomes a + o, the upper o - a, both as one fused
    // multiply-add with the lane's sign (exact products, one rounding: the
    // same values as the addition and the subtraction)
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float sgn_m = (lane & m) ? -1.f : 1.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, a[e], m);
        a[e] = fmaf(a[e], sgn_m, o);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      xr[r][e] = a[e] * inv_sqrt_d;
      amax = fmaxf(amax, fabsf(xr[r][e]));
    }
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
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int row = blk * 128 + warp * kRows + r;
    if (row < N)
      *reinterpret_cast<uint32_t*>(x8 + ((size_t)bh * N + row) * D + lane * E) =
          pack_e4m3x4(xr[r][0] * inv, xr[r][1] * inv, xr[r][2] * inv, xr[r][3] * inv);
  }
  if (threadIdx.x == 0) scales[(size_t)bh * nblk + blk] = scale;
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
