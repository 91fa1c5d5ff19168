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

// Q or K: rotate and quantise one 128-row block of one (batch, head) per CTA.
// 256 threads = 8 warps x 16 rows; a row is 32 lanes x 4 consecutive channels.
// The rotation is a fast Walsh-Hadamard transform: butterflies (a, b) ->
// (a + b, a - b) at strides 1 and 2 inside a lane, 4 ... 64 across lanes.
__global__ void __launch_bounds__(256)
    fa_fp8_rotate_quant_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs,
                               uint8_t* __restrict__ x8, float* __restrict__ scales, int N, int nblk) {
  constexpr int D = 128, E = 4, kRows = 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x, bh = blockIdx.y;
  __shared__ float red[8];
  float sgn[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sgn[e] = (float)signs[lane * E + e];
  const float inv_sqrt_d = 0.08838834764831845f;  // 1 / sqrt(128)
  float v[kRows][E];
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
    // strides 4 .. 64: the partner element sits in lane ^ (stride / 4)
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool upper = lane & m;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, a[e], m);
        a[e] = upper ? o - a[e] : a[e] + o;
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      v[r][e] = a[e] * inv_sqrt_d;
      amax = fmaxf(amax, fabsf(v[r][e]));
    }
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? amax / kE4m3Max : 1.f;
  const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int row = blk * 128 + warp * kRows + r;
    if (row < N)
      *reinterpret_cast<uint32_t*>(x8 + ((size_t)bh * N + row) * D + lane * E) =
          pack_e4m3x4(v[r][0] * inv, v[r][1] * inv, v[r][2] * inv, v[r][3] * inv);
  }
  if (threadIdx.x == 0) scales[(size_t)bh * nblk + blk] = scale;
}

// V, pass 1: per-channel maximum of |v| over one key block, folded into
// amax_bits[bh][c] (non-negative floats order like their bit patterns).
// 128 threads, thread = channel.
__global__ void __launch_bounds__(128)
    fa_fp8_v_amax_kernel(const __nv_bfloat16* __restrict__ v, unsigned* __restrict__ amax_bits, int N) {
  constexpr int D = 128;
  const int c = threadIdx.x, blk = blockIdx.x, bh = blockIdx.y;
  const int rows = min(128, N - blk * 128);
  const __nv_bfloat16* src = v + ((size_t)bh * N + blk * 128) * D + c;
  float m = 0.f;
  for (int r = 0; r < rows; ++r) m = fmaxf(m, fabsf(__bfloat162float(src[(size_t)r * D])));
  atomicMax(amax_bits + (size_t)bh * D + c, __float_as_uint(m));
}

// V, pass 2: quantise one key block per channel and write it transposed:
// v8t[bh][blk][c][key] (keys past N as zeros); the j = 0 block also writes the
// channel scales.  128 threads, thread = channel, holding its 128 keys as 32
// words of four E4M3 values and storing them as one 128-byte row.
__global__ void __launch_bounds__(128)
    fa_fp8_v_quant_kernel(const __nv_bfloat16* __restrict__ v, const unsigned* __restrict__ amax_bits,
                          uint8_t* __restrict__ v8t, float* __restrict__ v_scale, int N, int nblk) {
  constexpr int D = 128;
  const int c = threadIdx.x, blk = blockIdx.x, bh = blockIdx.y;
  const float amax = __uint_as_float(amax_bits[(size_t)bh * D + c]);
  const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
  const __nv_bfloat16* src = v + ((size_t)bh * N + blk * 128) * D + c;
  uint4* dst = reinterpret_cast<uint4*>(v8t + (((size_t)bh * nblk + blk) * D + c) * 128);
#pragma unroll 1
  for (int q = 0; q < 8; ++q) {  // 16 keys per 16-byte store
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = blk * 128 + 16 * q + 4 * i + e;
        f[e] = key < N ? __bfloat162float(src[(size_t)(16 * q + 4 * i + e) * D]) * inv : 0.f;
      }
      w[i] = pack_e4m3x4(f[0], f[1], f[2], f[3]);
    }
    dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (blk == 0) v_scale[(size_t)bh * D + c] = amax > 0.f ? amax / kE4m3Max : 1.f;
}

}  // namespace fa
