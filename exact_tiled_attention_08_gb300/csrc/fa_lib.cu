// C-ABI entry points of the exact tiled attention library (declared in fa.h).
//
// Host side only: argument validation, TMA tensor-map encoding and kernel
// launches.  All kernels live in the headers included below and are compiled
// into this one translation unit, which keeps the device status word a
// single per-device variable.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fa.h"
#include "sm103_ptx.cuh"
#include "fa_fwd.cuh"
#include "fa_bwd.cuh"
#include "fa_bwd_dq.cuh"
#include "fa_bwd_pair.cuh"
#include "fa_fp8.cuh"

namespace {

std::atomic<unsigned long long> g_wait_limit_ns{0};
std::atomic<int> g_debug_stall{0};
std::atomic<int> g_exp2_soft_quarters{0};
std::atomic<int> g_bwd_pair_mma{0};

// caller-owned events recorded around the main kernels (profiling hook)
struct TimingEvents {
  cudaEvent_t fwd_start = nullptr, fwd_stop = nullptr, bwd_start = nullptr, bwd_stop = nullptr;
};
std::mutex g_timing_mu;
TimingEvents g_timing;

TimingEvents timing_events() {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  return g_timing;
}
constexpr unsigned long long kDefaultWaitLimitNs = 10000ull * 1000 * 1000;

unsigned long long wait_limit_ns() {
  const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : kDefaultWaitLimitNs;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [B*H][N][d] bf16 viewed as a 3-D tensor (d, N, B*H); boxes of 64 x box_rows
// rows (128 by default), 128-byte swizzle.  Rows past N inside a head read as zero.
bool encode_bhnd(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bytes [outer][rows][inner] viewed as a 3-D tensor (inner, rows, outer); boxes of
// 128 bytes x 128 rows, 128-byte swizzle.  Rows past `rows` read as zero.
bool encode_u8_3d(CUtensorMap* map, const void* ptr, int inner, int rows, long long outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  const cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)inner * rows};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// shape checks shared by every entry point.  Sizes arrive as int; the
// kernels address memory with 64-bit offsets and count their work items
// (128-row blocks of every (batch, head), and the forward's pairs of them) in
// int, so B * H and (ceil(N / 128) + 1) * B * H must stay below 2^31.  That
// bounds B * H * N * d by 2^45 elements, far beyond the device's memory.
fa_status check_shape(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = (long long)B * H;
  if (bh > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  const long long blocks = ((long long)N + 127) / 128;
  if ((blocks + 1) * bh > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Every tensor argument must be memory the current device's kernels can read
// and write: device memory of the current device, or managed memory.  Host
// memory, another device's memory and addresses no allocation covers are
// refused before anything is enqueued (a kernel given one would fault).
fa_status check_device_ptrs(std::initializer_list<const void*> ptrs) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  for (const void* ptr : ptrs) {
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
      cudaGetLastError();  // leave no error behind for the launch checks that follow
      return e == cudaErrorInvalidValue ? FA_ERR_INVALID_ARG : FA_ERR_CUDA;
    }
    if (a.type == cudaMemoryTypeManaged) continue;
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

fa_status check_scale(float scale, int causal) {
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

template <typename Kernel>
cudaError_t set_smem(Kernel kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, bool CAUSAL, bool FP8 = false, int SOFT_EXP = 0>
fa_status launch_fwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, fa::FwdParams p,
                     int BH, cudaStream_t stream) {
  using C = fa::FwdCfg<D, FP8>;
  auto kernel = fa::fa_fwd_kernel<D, CAUSAL, FP8, SOFT_EXP>;
  if (set_smem(kernel, C::kSmemBytes) != cudaSuccess) return FA_ERR_CUDA;
  // the warpgroups re-divide the block's registers (setmaxnreg); that only
  // works if the block really gets kLaunchRegs per thread
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess || attr.numRegs != C::kLaunchRegs) return FA_ERR_CUDA;
  // persistent CTAs: one per SM (the kernel holds a whole SM), never more than there are items
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return FA_ERR_CUDA;
  // Without the mask all pairs cost the same, and a last round of rem < sms
  // pairs would keep the other SMs idle for a whole pair's time: when the
  // pairs of that round fit on the SMs as single tiles, they run as single
  // tiles.  (With the mask the last ranks are the lightest pairs already.)
  const int pairs = p.num_pairs * BH;
  const int rem = pairs % sms;
  p.pair_items = (!CAUSAL && rem > 0 && 2 * rem <= sms) ? pairs - rem : pairs;
  p.num_items = p.pair_items + 2 * (pairs - p.pair_items);
  const long long grid = p.num_items < sms ? p.num_items : sms;
  const TimingEvents ev = timing_events();
  if (ev.fwd_start && ev.fwd_stop && cudaEventRecord(ev.fwd_start, stream) != cudaSuccess) return FA_ERR_CUDA;
  kernel<<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (ev.fwd_start && ev.fwd_stop && cudaEventRecord(ev.fwd_stop, stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

// Heads per group of the causal item order of the backward kernels: the
// smallest divisor of the head count whose group holds at least four times
// the SMs' worth of the costliest item (need = ceil(4 sms / (nblk + 1))
// heads, so that a group's costliest items, handed out first, finish well
// before the group's one-block items run out), or all heads.  Groups of few
// heads keep the working set (their Q and dO, or K and V) small enough for
// L2.  Divisors come in pairs (i, BH / i), so i up to sqrt(BH) finds them all.
int causal_group_heads(int BH, int nblk, int sms) {
  const long long need = (4LL * sms + nblk) / (nblk + 1);
  long long best = BH;
  for (long long i = 1; i * i <= BH; ++i) {
    if (BH % i) continue;
    const long long j = BH / i;
    if (i >= need && i < best) best = i;
    if (j >= need && j < best) best = j;
  }
  return (int)best;
}

template <int D, bool CAUSAL, bool ATOMIC_DQ>
fa_status launch_bwd(const CUtensorMap* maps, const fa::BwdParams& p, int BH, cudaStream_t stream) {
  using C = fa::BwdCfg<D, ATOMIC_DQ>;
  auto kernel = fa::fa_bwd_kernel<D, CAUSAL, ATOMIC_DQ>;
  if (set_smem(kernel, C::kSmemBytes) != cudaSuccess) return FA_ERR_CUDA;
  // the kernel's warpgroups re-divide the registers the block launches with
  // (setmaxnreg); that only works if the block really gets 128 per thread
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess || attr.numRegs != C::kLaunchRegs) return FA_ERR_CUDA;
  // Without the mask every (key block, head) item costs the same: persistent
  // CTAs, one per SM, walk the items, and each overlaps one item's last dQ
  // reduction and dK/dV write with the next item's K/V load and first
  // products.  With the mask the items' costs range from 1 to nkb query
  // blocks, and one CTA per item lets the hardware balance them.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return FA_ERR_CUDA;
  fa::BwdParams q = p;
  q.num_items = p.nkb * BH;
  q.num_bh = BH;
  q.group_heads = causal_group_heads(BH, p.nkb, sms);
  const long long grid = (!CAUSAL && q.num_items > sms) ? sms : q.num_items;
  const TimingEvents ev = timing_events();
  if (ev.bwd_start && ev.bwd_stop && cudaEventRecord(ev.bwd_start, stream) != cudaSuccess) return FA_ERR_CUDA;
  kernel<<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                                                                  maps[8], q);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  if (ev.bwd_start && ev.bwd_stop && cudaEventRecord(ev.bwd_stop, stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

// dK/dV of the deterministic backward on CTA pairs (fa_bwd_pair.cuh, d = 128):
// clusters of two CTAs on adjacent key blocks, persistent without the mask
// (as many pairs as fit at once), one pair per item with it.
template <bool CAUSAL>
fa_status launch_bwd_pair(const CUtensorMap* maps, const fa::BwdParams& p, int BH, cudaStream_t stream) {
  using C = fa::BwdPairCfg;
  auto kernel = fa::fa_bwd_pair_kernel<CAUSAL>;
  if (set_smem(kernel, C::kSmemBytes) != cudaSuccess) return FA_ERR_CUDA;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess || attr.numRegs != C::kLaunchRegs) return FA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 2)
    return FA_ERR_CUDA;
  fa::BwdParams q = p;
  const int nj = (p.nkb + 1) / 2;  // pairs of key blocks per head
  q.num_items = nj * BH;
  q.num_bh = BH;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute cluster_attr[1];
  cluster_attr[0].id = cudaLaunchAttributeClusterDimension;
  cluster_attr[0].val.clusterDim.x = 2;
  cluster_attr[0].val.clusterDim.y = 1;
  cluster_attr[0].val.clusterDim.z = 1;
  cfg.attrs = cluster_attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.gridDim = dim3(2 * (unsigned)(sms / 2), 1, 1);
  int pairs = 0;
  if (cudaOccupancyMaxActiveClusters(&pairs, kernel, &cfg) != cudaSuccess || pairs < 1) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  q.group_heads = causal_group_heads(BH, nj, pairs);
  const long long units = (!CAUSAL && q.num_items > pairs) ? pairs : q.num_items;
  cfg.gridDim = dim3((unsigned)(2 * units), 1, 1);
  const TimingEvents ev = timing_events();
  if (ev.bwd_start && ev.bwd_stop && cudaEventRecord(ev.bwd_start, stream) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], q) !=
      cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  if (ev.bwd_start && ev.bwd_stop && cudaEventRecord(ev.bwd_stop, stream) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

template <int D, bool CAUSAL>
fa_status launch_bwd_dq(const CUtensorMap* maps, const fa::BwdDqParams& p, int BH, cudaStream_t stream) {
  using C = fa::BwdDqCfg<D>;
  auto kernel = fa::fa_bwd_dq_kernel<D, CAUSAL>;
  if (set_smem(kernel, C::kSmemBytes) != cudaSuccess) return FA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return FA_ERR_CUDA;
  fa::BwdDqParams q = p;
  q.num_bh = BH;
  q.group_heads = causal_group_heads(BH, p.nqb, sms);
  const long long grid = (long long)p.nqb * BH;
  kernel<<<(unsigned)grid, C::kThreads, C::kSmemBytes, stream>>>(maps[0], maps[1], maps[2], maps[3], q);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// the fp32 dQ accumulator [B*H][N][d] viewed as a 3-D tensor (d, N, B*H); boxes
// of 32 x 32 rows, 128-byte swizzle (the backward's reducers add such tiles
// with TMA reduces; rows past N inside a head are not written)
bool encode_dq_acc(CUtensorMap* map, const float* ptr, int BH, int N, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows][cols] viewed as a 2-D tensor (cols, rows); boxes of box_cols x 1, no swizzle
bool encode_f32_rows(CUtensorMap* map, const void* ptr, int rows, int cols, int box_cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, 1};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// workspace of fa_bwd: fp32 dQ accumulator, then delta and LSE*log2(e) padded
// to whole 128-row blocks, each at a 256-byte boundary
struct BwdWorkspace {
  size_t dq_bytes, stat_bytes;
  static BwdWorkspace of(int B, int H, int N, int d) {
    const size_t rows = (size_t)B * H * N;
    const size_t npad = (size_t)((N + 127) / 128) * 128;
    BwdWorkspace w;
    w.dq_bytes = (rows * d * sizeof(float) + 255) & ~size_t(255);
    w.stat_bytes = ((size_t)B * H * npad * sizeof(float) + 255) & ~size_t(255);
    return w;
  }
  size_t total() const { return dq_bytes + 2 * stat_bytes; }
};

// workspace of fa_fwd_fp8: Q8, K8 [B*H][N][128] E4M3, V8^T [B*H][nkb][128][128]
// E4M3, query and key block scales [B*H][nkb] fp32, value channel maxima (as
// bits) and scales [B*H][128] fp32; each part on a 256-byte boundary
struct Fp8Workspace {
  size_t q8, k8, v8t, qs, ks, vamax, vs, total;
  static Fp8Workspace of(int B, int H, int N) {
    const size_t bh = (size_t)B * H, nkb = (size_t)((N + 127) / 128);
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    Fp8Workspace w;
    size_t o = 0;
    w.q8 = o;
    o += up(bh * N * 128);
    w.k8 = o;
    o += up(bh * N * 128);
    w.v8t = o;
    o += up(bh * nkb * 128 * 128);
    w.qs = o;
    o += up(bh * nkb * 4);
    w.ks = o;
    o += up(bh * nkb * 4);
    w.vamax = o;
    o += up(bh * 128 * 4);
    w.vs = o;
    o += up(bh * 128 * 4);
    w.total = o;
    return w;
  }
};

// The backward pass proper, given device scratch of BwdWorkspace::total() bytes.
// deterministic: dQ by the separate query-major pass instead of fp32 atomics
// (the dQ accumulator part of the scratch is then not used).
fa_status run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, void* scratch, int B, int H, int N, int d, float scale, int causal,
                  bool deterministic, cudaStream_t stream) {
  const int BH = B * H;
  const int nkb = (N + 127) / 128;
  const int npad = nkb * 128;
  const BwdWorkspace w = BwdWorkspace::of(B, H, N, d);
  float* dq_acc = deterministic ? nullptr : static_cast<float*>(scratch);
  float* delta_pad = reinterpret_cast<float*>(static_cast<char*>(scratch) + w.dq_bytes);
  float* lse2_pad = reinterpret_cast<float*>(static_cast<char*>(scratch) + w.dq_bytes + w.stat_bytes);
  // maps[6], maps[7]: Q and dO in boxes of 64 rows (the CTA-pair kernel's row halves);
  // maps[8]: the dQ accumulator (atomic dQ only; otherwise a copy of maps[0] that
  // nothing reads)
  CUtensorMap maps[9];
  if (!encode_bhnd(&maps[0], q, BH, N, d) || !encode_bhnd(&maps[1], k, BH, N, d) ||
      !encode_bhnd(&maps[2], v, BH, N, d) || !encode_bhnd(&maps[3], dout, BH, N, d) ||
      !encode_f32_rows(&maps[4], lse2_pad, BH, npad, 128) || !encode_f32_rows(&maps[5], delta_pad, BH, npad, 128) ||
      !encode_bhnd(&maps[6], q, BH, N, d, 64) || !encode_bhnd(&maps[7], dout, BH, N, d, 64))
    return FA_ERR_CUDA;
  if (dq_acc && !encode_dq_acc(&maps[8], dq_acc, BH, N, d)) return FA_ERR_CUDA;
  if (!dq_acc) maps[8] = maps[0];
  // 1. delta, LSE*log2(e) (padded), dQ accumulator = 0 (atomic dQ only)
  {
    const long long padded_rows = (long long)BH * npad;
    const long long per_block = 256 / (d / 8);
    long long blocks = (padded_rows + per_block - 1) / per_block;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    if (d == 128)
      fa::fa_bwd_prep_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, delta_pad, lse2_pad,
          dq_acc, N, npad, padded_rows);
    else
      fa::fa_bwd_prep_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, delta_pad, lse2_pad,
          dq_acc, N, npad, padded_rows);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  }
  // 2. dK, dV (and the fp32 dQ accumulation)
  fa::BwdParams p;
  p.dq_acc = dq_acc;
  p.dk_out = static_cast<__nv_bfloat16*>(dk);
  p.dv_out = static_cast<__nv_bfloat16*>(dv);
  p.N = N;
  p.nkb = nkb;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.scale = scale;
  p.wait_limit_ns = wait_limit_ns();
  p.debug_stall = g_debug_stall.load();
  p.out_align32 = aligned32(dk) && aligned32(dv);
  fa_status st;
  if (deterministic) {
    if (d == 128 && g_bwd_pair_mma.load())
      st = causal ? launch_bwd_pair<true>(maps, p, BH, stream) : launch_bwd_pair<false>(maps, p, BH, stream);
    else if (d == 128)
      st = causal ? launch_bwd<128, true, false>(maps, p, BH, stream) : launch_bwd<128, false, false>(maps, p, BH, stream);
    else
      st = causal ? launch_bwd<64, true, false>(maps, p, BH, stream) : launch_bwd<64, false, false>(maps, p, BH, stream);
    if (st != FA_OK) return st;
    // 3'. dQ by the query-major pass, written once as bf16
    fa::BwdDqParams pq;
    pq.delta_pad = delta_pad;
    pq.lse2_pad = lse2_pad;
    pq.dq = static_cast<__nv_bfloat16*>(dq);
    pq.N = N;
    pq.nqb = nkb;
    pq.scale_log2 = p.scale_log2;
    pq.scale = scale;
    pq.wait_limit_ns = p.wait_limit_ns;
    pq.debug_stall = p.debug_stall;
    if (d == 128)
      return causal ? launch_bwd_dq<128, true>(maps, pq, BH, stream) : launch_bwd_dq<128, false>(maps, pq, BH, stream);
    return causal ? launch_bwd_dq<64, true>(maps, pq, BH, stream) : launch_bwd_dq<64, false>(maps, pq, BH, stream);
  }
  if (d == 128)
    st = causal ? launch_bwd<128, true, true>(maps, p, BH, stream) : launch_bwd<128, false, true>(maps, p, BH, stream);
  else
    st = causal ? launch_bwd<64, true, true>(maps, p, BH, stream) : launch_bwd<64, false, true>(maps, p, BH, stream);
  if (st != FA_OK) return st;
  // 3. dQ = scale * dQ_acc -> bf16
  const long long n8 = (long long)BH * N * d / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  fa::fa_dq_convert_kernel<<<(unsigned)blocks, 256, 0, stream>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), scale, n8);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status launch_preprocess(const void* o, const void* dout, float* delta, float* dq_acc, long long rows, int d,
                            cudaStream_t stream) {
  const long long per_block = 256 / (d / 8);
  long long blocks = (rows + per_block - 1) / per_block;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (d == 128)
    fa::fa_bwd_preprocess_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta, dq_acc, rows);
  else
    fa::fa_bwd_preprocess_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta, dq_acc, rows);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

void fa_set_wait_limit_ns(unsigned long long limit_ns) { g_wait_limit_ns.store(limit_ns); }

void fa_debug_stall(int enable) { g_debug_stall.store(enable ? 1 : 0); }

void fa_set_bwd_pair_mma(int enable) { g_bwd_pair_mma.store(enable ? 1 : 0); }

fa_status fa_set_exp2_split(int soft_quarters) {
  if (soft_quarters < 0 || soft_quarters > 2) return FA_ERR_INVALID_ARG;
  g_exp2_soft_quarters.store(soft_quarters);
  return FA_OK;
}

void fa_set_timing_events(cudaEvent_t fwd_start, cudaEvent_t fwd_stop, cudaEvent_t bwd_start, cudaEvent_t bwd_stop) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing.fwd_start = fwd_start;
  g_timing.fwd_stop = fwd_stop;
  g_timing.bwd_start = bwd_start;
  g_timing.bwd_stop = bwd_stop;
}

fa_status fa_check_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_fa_device_status, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_device_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return static_cast<fa_status>(word & 0xffu);
  }
  return FA_OK;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale, causal)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  if ((st = check_device_ptrs({q, k, v, o, lse})) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhnd(&mq, q, BH, N, d) || !encode_bhnd(&mk, k, BH, N, d) || !encode_bhnd(&mv, v, BH, N, d))
    return FA_ERR_CUDA;
  fa::FwdParams p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_align32 = aligned32(o);
  p.lse = lse;
  p.N = N;
  p.num_pairs = (N + 255) / 256;
  p.num_bh = BH;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.debug_stall = g_debug_stall.load();
  switch (g_exp2_soft_quarters.load()) {
    case 1:
      if (d == 128)
        return causal ? launch_fwd<128, true, false, 1>(mq, mk, mv, p, BH, stream)
                      : launch_fwd<128, false, false, 1>(mq, mk, mv, p, BH, stream);
      return causal ? launch_fwd<64, true, false, 1>(mq, mk, mv, p, BH, stream)
                    : launch_fwd<64, false, false, 1>(mq, mk, mv, p, BH, stream);
    case 2:
      if (d == 128)
        return causal ? launch_fwd<128, true, false, 2>(mq, mk, mv, p, BH, stream)
                      : launch_fwd<128, false, false, 2>(mq, mk, mv, p, BH, stream);
      return causal ? launch_fwd<64, true, false, 2>(mq, mk, mv, p, BH, stream)
                    : launch_fwd<64, false, false, 2>(mq, mk, mv, p, BH, stream);
    default:
      if (d == 128)
        return causal ? launch_fwd<128, true>(mq, mk, mv, p, BH, stream) : launch_fwd<128, false>(mq, mk, mv, p, BH, stream);
      return causal ? launch_fwd<64, true>(mq, mk, mv, p, BH, stream) : launch_fwd<64, false>(mq, mk, mv, p, BH, stream);
  }
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d) != FA_OK || d != 128) return 0;
  return Fp8Workspace::of(B, H, N).total;
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, const signed char* signs, void* o, float* lse,
                     void* workspace, size_t ws_bytes, int B, int H, int N, int d, float scale, int causal,
                     cudaStream_t stream) {
  if (!q || !k || !v || !signs || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale, causal)) != FA_OK) return st;
  if (ws_bytes < fa_fwd_fp8_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
    return FA_ERR_MISALIGNED;
  // the V quantisation's grid has one y index per (batch, head)
  if ((long long)B * H > 65535) return FA_ERR_UNSUPPORTED;
  if ((st = check_device_ptrs({q, k, v, signs, o, lse, workspace})) != FA_OK) return st;
  const int BH = B * H;
  const int nkb = (N + 127) / 128;
  const Fp8Workspace w = Fp8Workspace::of(B, H, N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* q8 = ws + w.q8;
  uint8_t* k8 = ws + w.k8;
  uint8_t* v8t = ws + w.v8t;
  float* qs = reinterpret_cast<float*>(ws + w.qs);
  float* ks = reinterpret_cast<float*>(ws + w.ks);
  unsigned* vamax = reinterpret_cast<unsigned*>(ws + w.vamax);
  float* vs = reinterpret_cast<float*>(ws + w.vs);
  // 1. operands: rotate and quantise Q, K per block; V per channel, transposed
  const dim3 grid_rows((unsigned)nkb, (unsigned)BH);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  const int8_t* sg = reinterpret_cast<const int8_t*>(signs);
  if (cudaMemsetAsync(vamax, 0, (size_t)BH * 128 * sizeof(unsigned), stream) != cudaSuccess) return FA_ERR_CUDA;
  CUtensorMap mxq, mxk, mxv;
  if (!encode_bhnd(&mxq, q, BH, N, 128) || !encode_bhnd(&mxk, k, BH, N, 128) || !encode_bhnd(&mxv, v, BH, N, 128))
    return FA_ERR_CUDA;
  if (set_smem(fa::fa_fp8_prepare_kernel, fa::kFp8PrepSmemBytes) != cudaSuccess) return FA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return FA_ERR_CUDA;
  const long long prep_items = 3LL * BH * nkb;
  const long long prep_cap = (long long)sms * fa::kFp8PrepCtasPerSm;
  const long long prep_grid = prep_items < prep_cap ? prep_items : prep_cap;
  CUtensorMap mq, mk, mv;
  if (!encode_u8_3d(&mq, q8, 128, N, BH) || !encode_u8_3d(&mk, k8, 128, N, BH) ||
      !encode_u8_3d(&mv, v8t, 128, 128, (long long)BH * nkb))
    return FA_ERR_CUDA;
  fa::fa_fp8_prepare_kernel<<<(unsigned)prep_grid, fa::kFp8PrepThreads, fa::kFp8PrepSmemBytes, stream>>>(
      mxq, mxk, mxv, mq, mk, sg, qs, ks, vamax, N, nkb, BH, wait_limit_ns());
  fa::fa_fp8_v_quant_kernel<<<grid_rows, 256, 0, stream>>>(vb, vamax, v8t, vs, N, nkb);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  // 2. attention on the E4M3 operands
  fa::FwdParams p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_align32 = aligned32(o);
  p.lse = lse;
  p.N = N;
  p.num_pairs = (N + 255) / 256;
  p.num_bh = BH;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.debug_stall = g_debug_stall.load();
  p.q_scale = qs;
  p.k_scale = ks;
  p.v_scale = vs;
  p.nkb = nkb;
  return causal ? launch_fwd<128, true, true>(mq, mk, mv, p, BH, stream)
                : launch_fwd<128, false, true>(mq, mk, mv, p, BH, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d) != FA_OK) return 0;
  return BwdWorkspace::of(B, H, N, d).total();
}

fa_status fa_bwd_preprocess(const void* o, const void* dout, float* delta, int B, int H, int N, int d,
                            cudaStream_t stream) {
  if (!o || !dout || !delta) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(delta)) return FA_ERR_MISALIGNED;
  if ((st = check_device_ptrs({o, dout, delta})) != FA_OK) return st;
  return launch_preprocess(o, dout, delta, nullptr, (long long)B * H * N, d, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                 float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale, causal)) != FA_OK) return st;
  if (ws_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return FA_ERR_MISALIGNED;
  if ((st = check_device_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace})) != FA_OK) return st;
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, H, N, d, scale, causal, false, stream);
}

fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                               int B, int H, int N, int d, float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale, causal)) != FA_OK) return st;
  if (ws_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return FA_ERR_MISALIGNED;
  if ((st = check_device_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace})) != FA_OK) return st;
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, H, N, d, scale, causal, true, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward with library-owned scratch, for callers that cannot allocate.
//
// fa_bwd needs an fp32 dQ accumulator and the delta vector in device memory
// that the caller provides.  Some callers cannot provide it when they call
// the backward: code running inside a runtime that owns all device memory
// through its own arena and does not let plug-ins call cudaMalloc while it
// executes, or code that must keep a fixed device-memory footprint once it
// has started.  fa_bwd_static_scratch takes its scratch from the file-scope
// array below instead, whose size is fixed when the library is loaded: every
// device that loads the library holds these FA_STATIC_SCRATCH_BYTES until
// the process exits, and no call allocates anything.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_fa_static_scratch[FA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
void* g_static_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
fa_status static_scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_static_scratch_mu);
  if (!g_static_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_static_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_static_scratch_ptr[dev] = p;
  }
  *out = g_static_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                float scale, int causal, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  fa_status st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale, causal)) != FA_OK) return st;
  if (fa_bwd_workspace_bytes(B, H, N, d) > (size_t)FA_STATIC_SCRATCH_BYTES) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  if ((st = check_device_ptrs({q, k, v, o, dout, lse, dq, dk, dv})) != FA_OK) return st;
  void* scratch = nullptr;
  if ((st = static_scratch_on_current_device(&scratch)) != FA_OK) return st;
  // the previous call's contents stay in the array: the preprocess rewrites
  // delta and LSE*log2(e) and zeroes the dQ accumulator before anything reads them
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, B, H, N, d, scale, causal, false, stream);
}

}  // extern "C"
