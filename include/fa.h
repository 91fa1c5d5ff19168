/*
 * fa.h - C ABI of the exact tiled attention library for GB300 (sm_103a).
 *
 * The library computes exact softmax attention, O = softmax(scale * Q K^T) V,
 * without ever writing an N x N matrix to device memory:
 *
 *   - the forward pass keeps a block of 128 queries on chip and streams the
 *     keys and values past it in blocks of 128 with the online softmax
 *     (running maximum m, running sum l = sum e^{s-m}, rescaled output
 *     accumulator), then writes O and one log-sum-exp L_i = m_i + log l_i per
 *     query row ("Interrogating the GPU part 5: FlashAttention", sections
 *     "How does tiling remove the traffic?" and "How can you softmax a row you
 *     never see whole?", online-softmax update equation; "LLM Flash
 *     Attention", section "End-to-end flow");
 *   - the backward pass recomputes every probability tile as
 *     P_ij = exp(S_ij - L_i) from Q, K and the saved L, and forms
 *     dV = P^T dO, dS = P o (dP - delta), dQ = scale dS K, dK = scale dS^T Q
 *     ("Interrogating the GPU part 5: FlashAttention", section "What does the
 *     backward pass do without P?", LSE equation and recompute formula).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  Q, K, V, O, dO, dQ, dK, dV are contiguous bf16 arrays laid out
 *   [B][H][N][d] (row-major, d fastest).  LSE and delta are contiguous fp32
 *   arrays [B][H][N].  Queries and keys share the length N.
 * Scores.  S = scale * Q K^T; LSE is in natural-log units of the scaled scores.
 * Causal.  causal = 1 hides key j from query i when j > i (top-left aligned);
 *   causal = 0 attends to all N keys.
 * Memory.  Every pointer is device memory owned by the caller; the library
 *   allocates nothing (no cudaMalloc; tensor memory is taken and released
 *   inside each thread block).  Its only state is one device status word per
 *   device, used to report a kernel that gave up waiting (FA_ERR_TIMEOUT).
 * Streams.  Calls only enqueue work on `stream` (0 = legacy default stream) and
 *   return the launch status; they do not synchronize.  A device-side timeout
 *   is reported later by fa_check_device_status.
 * Device.  Every call runs on the CURRENT device (cudaGetDevice): the caller
 *   makes the tensors' device current first.  Every tensor pointer must be
 *   device memory of that device, or managed memory; anything else (host
 *   memory, another device's memory, an address no allocation covers) gives
 *   FA_ERR_INVALID_ARG before anything is enqueued.
 * Errors.  Arguments are validated before anything is enqueued; on an error
 *   nothing runs and no output is written.  Invalid sizes, a null pointer, a
 *   pointer the current device cannot use (above) or a non-finite /
 *   non-positive scale give FA_ERR_INVALID_ARG; a pointer not on a 16-byte
 *   boundary gives FA_ERR_MISALIGNED; a head dimension other than 64 or 128
 *   gives FA_ERR_UNSUPPORTED; a failed CUDA call (including a device without
 *   sm_103a support) gives FA_ERR_CUDA.
 * Validity of the outputs.  A returned FA_OK means the work was enqueued.
 *   Every wait inside the kernels is bounded in time (fa_set_wait_limit_ns,
 *   default 10 s); a kernel whose wait runs out -- which also happens if the
 *   GPU stops running it for longer than the limit, e.g. under heavy time
 *   slicing -- stops early, leaves its outputs undefined and records
 *   FA_ERR_TIMEOUT in the device status word.  The outputs of a sequence of
 *   calls are therefore known to be valid only once fa_check_device_status
 *   has returned FA_OK after them.
 * Limits.  1 <= B, H, N; B * H < 2^31 and (ceil(N / 128) + 1) * B * H < 2^31
 *   (the kernels count 128-row blocks in 32-bit integers and address memory
 *   with 64-bit offsets, so B * H * N * d itself may exceed 2^31);
 *   fa_fwd_fp8 also needs B * H <= 65535.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_MISALIGNED = 2,
  FA_ERR_UNSUPPORTED = 3,
  FA_ERR_CUDA = 4,
  FA_ERR_TIMEOUT = 5
} fa_status;

/*
 * Forward pass.  "Interrogating the GPU part 5: FlashAttention", sections
 * "How does tiling remove the traffic?" and "How can you softmax a row you
 * never see whole?" (online-softmax update equation), with the log-sum-exp
 * of section "What does the backward pass do without P?"; causal block
 * skipping as in "LLM Flash Attention", section "End-to-end flow".
 *
 *   q, k, v  in:  bf16 [B][H][N][d]
 *   o        out: bf16 [B][H][N][d], O = softmax(scale Q K^T) V
 *   lse      out: fp32 [B][H][N],   L_i = log sum_j exp(scale q_i . k_j)
 *   scale    finite, > 0 (1/sqrt(d) for standard attention)
 *   causal   0 or 1
 *   d        64 or 128
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, cudaStream_t stream);

/*
 * FP8 forward.  "Interrogating the GPU part 5: FlashAttention", section "What
 * did FlashAttention-3 do with Hopper?" (FP8 quantised per block after a
 * random Hadamard rotation, which spreads outliers across the block);
 * "FlashAttention versions", section "FlashAttention-3 (2024)" (block-level
 * quantisation instead of one per-tensor scale).  Same result as fa_fwd up
 * to FP8 rounding, with the products on the tensor cores' E4M3 path:
 *   1. Q and K rows are rotated by R = diag(signs) H / sqrt(128) (H the
 *      Sylvester Hadamard matrix), which leaves Q K^T unchanged, and rounded
 *      to E4M3 (nearest even, saturating at +-448) with one scale per block
 *      of 128 rows of each (batch, head): scale = max|x R| / 448;
 *   2. V is rounded to E4M3 with one scale per channel of each (batch, head)
 *      over the sequence: scale = max_n |v_nc| / 448;
 *   3. the online softmax of fa_fwd runs on the dequantised scores, the
 *      probabilities are rounded to E4M3 for the P V product, and O is
 *      normalised by the sum of the rounded probabilities and multiplied by
 *      the value channel scales.  LSE uses the unrounded sum.
 *
 *   q, k, v    in:  bf16 [B][H][N][128]
 *   signs      in:  int8 [128] device array of +1 / -1 (the random signs of
 *                   the rotation; the caller draws them)
 *   o, lse     out: as for fa_fwd
 *   workspace  device scratch of ws_bytes >= fa_fwd_fp8_workspace_bytes(),
 *              16-byte aligned.  Layout (each part on a 256-byte boundary,
 *              in this order): Q R and K R in E4M3 [B][H][N][128];
 *              V^T in E4M3 [B][H][nkb][128 channels][128 keys] (keys past N
 *              zero), nkb = ceil(N / 128); query and key block scales fp32
 *              [B][H][nkb] each; value channel maxima (fp32 bits) and scales
 *              fp32 [B][H][128] each.  Its contents on entry are ignored.
 *   d          128 only (other values give FA_ERR_UNSUPPORTED)
 */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d);
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, const signed char* signs, void* o, float* lse,
                     void* workspace, size_t ws_bytes, int B, int H, int N, int d, float scale, int causal,
                     cudaStream_t stream);

/*
 * Backward preprocess: delta_i = sum_c dO_ic * O_ic, one fp32 per query row.
 * The term delta of dS = P o (dP - delta) in "Interrogating the GPU part 5:
 * FlashAttention", section "What does the backward pass do without P?"; the
 * pages do not define it, and the row sum of dO o O is its exact value
 * (sum_j P_ij dP_ij with dP = dO V^T and O = P V).
 *
 *   o, dout  in:  bf16 [B][H][N][d]
 *   delta    out: fp32 [B][H][N]
 */
fa_status fa_bwd_preprocess(const void* o, const void* dout, float* delta, int B, int H, int N, int d,
                            cudaStream_t stream);

/*
 * Bytes of device workspace fa_bwd needs: an fp32 dQ accumulator
 * [B][H][N][d], then delta and LSE*log2(e) as fp32 [B][H][Npad] each, where
 * Npad = 128 * ceil(N / 128) (every part starting on a 256-byte boundary).
 * Returns 0 for sizes fa_bwd would reject.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass by recomputation.  "Interrogating the GPU part 5:
 * FlashAttention", section "What does the backward pass do without P?" (LSE
 * equation, recompute formula P_ij = exp(S_ij - L_i), dV = P^T dO,
 * dS = P o (dP - delta)); "LLM Flash Attention", section "End-to-end flow"
 * (backward paragraph).  dQ is accumulated in fp32 in the workspace and cast
 * to bf16 at the end.
 *
 *   q, k, v, o, dout  in:  bf16 [B][H][N][d]; o and lse as written by fa_fwd
 *   lse               in:  fp32 [B][H][N]
 *   dq, dk, dv        out: bf16 [B][H][N][d] (overwritten, not accumulated)
 *   workspace         device scratch of ws_bytes >= fa_bwd_workspace_bytes(),
 *                     16-byte aligned; its contents on entry are ignored
 *   scale, causal     as passed to fa_fwd
 * ws_bytes too small gives FA_ERR_INVALID_ARG.  dQ is summed with fp32
 * atomics, so it is not bitwise repeatable from run to run.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                 float scale, int causal, cudaStream_t stream);

/*
 * Backward pass with a deterministic dQ.  Same arguments, layout, workspace
 * (ws_bytes >= fa_bwd_workspace_bytes()) and error behaviour as fa_bwd, and
 * the same dQ, dK, dV up to rounding; dQ, dK and dV are bitwise repeatable
 * from run to run on the same device.  "Interrogating the GPU part 5:
 * FlashAttention", section "What does the backward pass do without P?"
 * (recompute formula, dS = P o (dP - delta)); "LLM Flash Attention", section
 * "End-to-end flow" (each recomputed block contributes to the gradients; how
 * the contributions to dQ are summed is left open).  Here they are summed by a
 * separate pass rather than with atomics: after the key-block-major pass that
 * forms dK and dV, a query-block-major pass recomputes S = Q K^T,
 * dP = dO V^T and dS for each of its query blocks, sums dQ = scale dS K over
 * the key blocks in a fixed order in tensor memory, and writes it once.
 * This costs three more N x N x d products per head pair (the backward does
 * 7 N^2 d multiply-adds per (batch, head) instead of 5) and needs no fp32
 * atomics; the dQ accumulator part of the workspace is not used.
 */
fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                               int B, int H, int N, int d, float scale, int causal, cudaStream_t stream);

/*
 * Backward pass with library-owned scratch.  This entry point has no
 * counterpart on the source pages; it exists for callers that cannot
 * allocate device memory when they run the backward pass -- for example a
 * plug-in inside a runtime that hands out device memory only from its own
 * arena and forbids cudaMalloc during execution, or a program that must keep
 * a fixed device-memory footprint after start-up.  It computes exactly what
 * fa_bwd computes, with the same arguments minus the workspace: the fp32 dQ
 * accumulator and delta live in a fixed array of FA_STATIC_SCRATCH_BYTES
 * compiled into the library, which every device that loads the library holds
 * until the process exits.  The call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *
 * Limit: shapes whose fa_bwd_workspace_bytes(B, H, N, d) exceeds
 * FA_STATIC_SCRATCH_BYTES (72 MiB; roughly B*H*N*(d+2)*4 bytes must fit, as
 * for B=4, H=16, N=2048, d=128) return FA_ERR_INVALID_ARG and run nothing.
 * Set-up: the first call on a device looks up the array's device address on
 * that device (cudaGetSymbolAddress, with that device current) and caches it
 * for the life of the process; make that first call outside any stream
 * capture.  The cached address belongs to the device's context: after
 * cudaDeviceReset (which destroys that context and the array with it) this
 * entry point must not be called again in the same process.  Sharing: every call uses
 * the same array and the array keeps the last call's contents (each call
 * re-initialises what it reads).  Calls whose work overlaps on the GPU (on
 * different streams, or from different threads) race on the array and give
 * wrong results; calls ordered on one stream do not.
 */
#define FA_STATIC_SCRATCH_BYTES (72u * 1024u * 1024u)
fa_status fa_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                float scale, int causal, cudaStream_t stream);

/*
 * Synchronizes `stream`, then returns and clears the current device's status
 * word: FA_OK, or FA_ERR_TIMEOUT if a kernel of this library gave up waiting
 * on one of its barriers since the last check (its outputs are then
 * undefined), or FA_ERR_CUDA if the synchronization itself failed.
 */
fa_status fa_check_device_status(cudaStream_t stream);

/*
 * Upper bound, in nanoseconds, on every barrier wait inside the kernels
 * launched after this call (process-wide; 0 restores the default of ten
 * seconds).  A wait that runs out makes the kernel stop early and report
 * FA_ERR_TIMEOUT through fa_check_device_status; it never traps.  Meant for
 * tests of that path.
 */
void fa_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * Test hook for the timeout path.  While `enable` is nonzero, every kernel
 * launched by fa_fwd / fa_bwd first makes its MMA-issuing thread wait on a
 * barrier that nothing ever signals; that wait runs out after the wait limit
 * (fa_set_wait_limit_ns), the kernel reports FA_ERR_TIMEOUT, drains the copies
 * it started and returns without writing its outputs.  Process-wide; 0 (the
 * default) turns it off.  Nothing traps or hangs.
 */
void fa_debug_stall(int enable);

/*
 * Where fa_fwd evaluates its exponentials ("Interrogating the GPU part 5:
 * FlashAttention", section "Why did Blackwell need FlashAttention-4?": part of
 * the exponentials run in software as 2^n times a cubic in the fraction, on
 * the FMA units, the rest on the special-function unit).  soft_quarters = 0
 * (the default) computes every probability with the special-function unit's
 * ex2; 1 or 2 computes that many of every four pairs of probabilities a
 * softmax thread forms with the cubic 1 + 0.6951 f + 0.2276 f^2 + 0.0771 f^3
 * (relative error <= 1.0e-4, 20 times below a bf16 probability's rounding).
 * The results stay within the same tolerances; only the speed differs.
 * Applies to the bf16 forward launched after the call (fa_fwd_fp8 always uses
 * the special-function unit).  Process-wide.  Other values give
 * FA_ERR_INVALID_ARG and change nothing.
 */
fa_status fa_set_exp2_split(int soft_quarters);

/*
 * How fa_bwd_deterministic forms dK and dV at d = 128 ("Interrogating the GPU
 * part 5: FlashAttention", section "Why did Blackwell need FlashAttention-4?":
 * the 2-SM MMA, in which two SMs compute one product of twice the rows, each
 * reading half of the other operand from its own shared memory).  enable = 0
 * (the default): one CTA per 128-key block, as fa_bwd.  enable != 0: clusters of
 * two CTAs on adjacent key blocks, whose four products per query block
 * (S^T, dP^T, dV, dK) run as 256-row tcgen05 MMAs across the pair; the
 * results are the same up to summation order and equally bitwise repeatable.
 * d = 64 and fa_bwd are not affected.  Process-wide; applies to calls made
 * after it.
 */
void fa_set_bwd_pair_mma(int enable);

/*
 * Profiling hook.  While set, fa_fwd and fa_fwd_fp8 record fwd_start and
 * fwd_stop on their stream immediately before and after launching the
 * attention kernel (not around fa_fwd_fp8's operand preparation), and fa_bwd
 * and fa_bwd_deterministic record bwd_start and bwd_stop around the main
 * backward kernel (not around the preprocess, the final dQ cast or the
 * deterministic dQ pass), so that cudaEventElapsedTime gives the duration of
 * exactly those kernels.  The events are created and
 * owned by the caller on the device the calls run on; a null pointer disables
 * its pair.  Process-wide; call again with nulls to turn it off.
 */
void fa_set_timing_events(cudaEvent_t fwd_start, cudaEvent_t fwd_stop, cudaEvent_t bwd_start,
                          cudaEvent_t bwd_stop);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
