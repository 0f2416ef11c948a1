/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library, libfa.so.
 *
 * The operation is exact scaled-dot-product attention computed tile by tile
 * with online softmax, so the N x N score and probability matrices never reach
 * device memory:
 *
 *     S = scale * Q K^T  (causal: S_ij = -inf for key j > query i),
 *     P = rowsoftmax(S),  O = P V,  lse_i = log sum_j exp(S_ij)
 *
 * ("FlashAttention-1", jshn9515 deep-learning-notes 10.2.1-10.2.3, for the
 * definition and the online-softmax rescaling; "Flash Attention V1/V2/V3演进",
 * sections V1分块原理 / 在线Softmax / V2并行优化, for tiling, the running
 * max/sum/output state and the one-time final normalisation; "5.4
 * FlashAttention", listing 3-1, for the alpha = exp(m_old - m_new) rescale.)
 * The backward recomputes P from the saved lse instead of storing it
 * ("FlashAttention-1", 10.2.4).
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, contiguous, row-major [B][H][N][d]; lse and delta are
 *     [B][H][N].  There are no strides.  Every device pointer must be 16-byte
 *     aligned (tensor-memory-accelerator copies need it); a misaligned pointer
 *     is FA_ERR_INVALID_ARG.
 *   - All pointers are DEVICE pointers on the current CUDA device unless a
 *     comment says otherwise.  The caller owns every buffer, including the
 *     backward workspace; the library allocates no device memory per call.  It
 *     owns only one status word per device, created on first use.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream: they enqueue kernels and
 *     return without synchronising.
 *   - Return value: an fa_status.  Argument problems are detected on the host
 *     before anything is launched.  Errors that happen inside a kernel (a
 *     bounded wait that ran out) are recorded in the per-device status word and
 *     reported by fa_last_device_error().
 *   - `scale` multiplies Q K^T (the configurations use 1/sqrt(d)).
 *   - Any N >= 1 is accepted (tiles past N are zero-filled and masked).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_F32 = 0, FA_BF16 = 1, FA_E4M3 = 2 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, N < 1, B/H < 1, bad dtype */
    FA_ERR_UNSUPPORTED = 2,     /* valid request this build does not implement      */
    FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call or launch failed      */
    FA_ERR_DEVICE_TIMEOUT = 4   /* a kernel's bounded wait ran out (device-side)    */
} fa_status;

/*
 * Size limits shared by every entry point: B*H (heads, or query heads) at most
 * 2^24, N (rows of one head) at most 2^24, and B*H*ceil(N/128) at most 2^31 - 1,
 * so that the kernels' work items (128-row blocks of one head) can be counted in
 * an int.  Larger sizes are refused with FA_ERR_UNSUPPORTED before anything runs.
 */

/*
 * Forward pass.  O = softmax(scale Q K^T [causal mask]) V and
 * lse_i = m_i + ln l_i (natural log, in units of the scaled score; m_i the row
 * max, l_i the row sum of exp(S_ij - m_i)), as on the "FlashAttention-1" page
 * 10.2.1 (standard attention, stable softmax) and 10.2.2 (online update).
 *
 *   q, k, v : [B][H][N][d] of `dtype`, read only.
 *   o       : [B][H][N][d] of `dtype`, written (fully overwritten).
 *   lse     : [B][H][N] float32, written.  May be NULL if not wanted.
 *   dtype   : FA_F32 (d = 64 or 128; exact fp32 CUDA-core kernel) or
 *             FA_BF16 (d = 64 or 128; tensor-core kernel with fp32
 *             accumulation; O rounded to bf16 to nearest even).
 *             FA_E4M3 is FA_ERR_INVALID_ARG here: use fa_fwd_fp8().
 *   causal  : 0 = full attention; 1 = key j attends only to queries i >= j.
 * Errors: FA_ERR_INVALID_ARG (null q/k/v/o, misalignment, B,H,N < 1, bad
 * dtype), FA_ERR_UNSUPPORTED (other d), FA_ERR_CUDA (launch failure).
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * FP8 forward ("Flash Attention V1/V2/V3演进", section V3增强: FP8 matrix
 * inputs, FP32 accumulation, scale factors).  Inputs are OCP E4M3 codes with
 * one float32 dequantisation factor per tensor: the real value of element x is
 * e4m3(x) * x_descale.  The kernel computes the same O and lse as fa_fwd on the
 * dequantised inputs; P is re-quantised to E4M3 inside the kernel for the P V
 * product (accumulation stays fp32).
 *
 *   q8, k8, v8 : [B][H][N][d] uint8 E4M3 codes.
 *   o          : [B][H][N][d] bfloat16, written.
 *   lse        : [B][H][N] float32, written (may be NULL).
 *   d          : 128.
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for a non-finite or <= 0 descale.
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse,
               float q_descale, float k_descale, float v_descale,
               int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Grouped-query forward: groups of H / H_kv query heads share one K/V head
 * (the "GQA" of the "5.4 FlashAttention" page's heading; the arithmetic per query
 * head is exactly fa_fwd's).  Query head h of batch b reads K/V head
 * b*H_kv + h / (H / H_kv).
 *
 *   q, o : [B][H][N][d] bfloat16;  k, v : [B][H_kv][N][d] bfloat16;  lse [B][H][N].
 *   dtype : FA_BF16.  d : 64 or 128.
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for H_kv < 1 or H % H_kv != 0;
 * FA_ERR_UNSUPPORTED for FA_F32.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int H_kv, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * FP8 forward with one dequantisation factor per (batch, head) instead of per
 * tensor: finer scale factors ("Flash Attention V1/V2/V3演进", section V3增强).
 * Element x of head (b, h) has the real value e4m3(x) * x_descale[b*H + h].
 *
 *   q_descale, k_descale, v_descale : DEVICE float32 arrays of B*H factors.
 *   Other arguments as fa_fwd_fp8.
 * Errors: as fa_fwd_fp8; FA_ERR_INVALID_ARG also for a null descale array.  The
 * factors themselves are read on the device and not validated.
 */
int fa_fwd_fp8_per_head(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                        const float* q_descale, const float* k_descale, const float* v_descale,
                        int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * FP8 forward with one dequantisation factor per 128-row block of each head, the
 * finest scale granularity here ("Flash Attention V1/V2/V3演进", section V3增强:
 * fine-grained scale factors).  Row i of head (b, h) of Q has the real value
 * e4m3(q8[b][h][i]) * q_descale[(b*H + h) * nb + i / 128], nb = ceil(N / 128), and the
 * same for K and V with their own arrays.  The result is the attention of the real
 * values, as fa_fwd_fp8.
 *
 *   q_descale, k_descale, v_descale : DEVICE float32 arrays of B*H*ceil(N/128)
 *                                     factors, positive and finite (read on the
 *                                     device, not validated).
 *   Other arguments as fa_fwd_fp8.
 * Method: the Q and K factors fold into the score constant per (query tile, key
 * block); V's factor for key block j scales P before its E4M3 rounding by
 * v_j / max_j v_j (at most 1), and the row sum and O are corrected exactly.
 * Errors: as fa_fwd_fp8_per_head.
 */
int fa_fwd_fp8_per_block(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                         const float* q_descale, const float* k_descale, const float* v_descale,
                         int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Forward over one shard of the keys, the per-shard step of sequence-sharded
 * attention: N_q queries at global positions q_offset + i against N_kv keys at
 * global positions kv_offset + j.  It is the forward of "FlashAttention-1",
 * 10.2.1-10.2.3, on the keys the shard holds; its normalised output and lse are
 * what fa_lse_merge combines across shards (the two-state combination of 10.2.2).
 *
 *   q        : [B][H][N_q][d] bfloat16.   k, v : [B][H_kv][N_kv][d] bfloat16
 *              (H_kv divides H; query head h reads K/V head h / (H / H_kv)).
 *   o_part   : [B][H][N_q][d] FLOAT32, written (the shard's normalised output).
 *   lse_part : [B][H][N_q] float32, written, required.
 *   causal   : 0, or 1: key j reaches query i iff kv_offset + j <= q_offset + i.
 *              A row that reaches no key of the shard gets O = 0, lse = -inf.
 *   dtype    : FA_BF16.  d : 64 or 128.  Offsets are only compared, never used
 *              to address memory: k and v start at the shard's first key.
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for lse_part null, N_kv < 1, or
 * H_kv not dividing H.
 */
int fa_fwd_kv_shard(const void* q, const void* k, const void* v, float* o_part,
                    float* lse_part, int B, int H, int H_kv, int N_q, int N_kv, int d,
                    float scale, int causal, long long q_offset, long long kv_offset,
                    int dtype, void* stream);

/*
 * Merge n_parts shard outputs of the same queries over disjoint key sets
 * ("FlashAttention-1", 10.2.2: partial states combine through their maxima and
 * sums; with normalised parts the weight of part s is exp(lse_s - lse)):
 *     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
 * Parts with lse_s = -inf add nothing; a row with every lse_s = -inf gives O = 0
 * and lse = -inf.  The result equals the forward over the union of the keys up to
 * rounding.
 *
 *   o_parts   : [n_parts][B][H][N][d] float32 (the fa_fwd_kv_shard outputs,
 *               stacked), read only.   lse_parts : [n_parts][B][H][N] float32.
 *   o         : [B][H][N][d] written, bfloat16 (dtype FA_BF16) or float32
 *               (FA_F32).   lse : [B][H][N] float32, written, or NULL.
 *   n_parts   : 1 to 16.   d : 64 or 128.  Every pointer 16-byte aligned.
 * Errors: FA_ERR_INVALID_ARG (null/misaligned pointers, n_parts < 1, bad sizes or
 * dtype), FA_ERR_UNSUPPORTED (other d, n_parts > 16), FA_ERR_CUDA (launch failure).
 */
int fa_lse_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o,
                 float* lse, int B, int H, int N, int d, int dtype, void* stream);

/*
 * Bytes of device workspace that fa_bwd needs for these sizes: the per-row
 * delta_i = dO_i . O_i and the pre-scaled lse (float32, N rounded up to 128
 * per head), plus for d = 64 the float32 dQ accumulator
 * ([B][H][N rounded up to 128][d]).
 * Returns 0 for invalid sizes and for sizes the backward refuses (beyond the
 * size limits above), whose byte count could overflow.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass by recomputation ("FlashAttention-1", 10.2.4): with
 * P_ij = exp(S_ij - lse_i) rebuilt tile by tile from the saved lse,
 *     dV = P^T dO,   dP = dO V^T,   delta_i = dO_i . O_i,
 *     dS = P o (dP - delta),   dQ = scale dS K,   dK = scale dS^T Q.
 *
 *   q, k, v, o, dO : [B][H][N][d] bfloat16, read only (o from fa_fwd).
 *   lse            : [B][H][N] float32 from fa_fwd, read only.
 *   dq, dk, dv     : [B][H][N][d] bfloat16, written.
 *   workspace      : device buffer of at least fa_bwd_workspace_size() bytes,
 *                    owned by the caller; its contents on entry do not matter
 *                    and on return are unspecified.  Calls that overlap in time
 *                    must not share one workspace.
 *   dtype          : FA_BF16.   d : 64 or 128 (d = 64 accumulates dQ with fp32
 *                    atomics in the workspace; d = 128 computes dQ in a second,
 *                    query-parallel kernel, and its workspace holds no accumulator).
 *   causal         : 0, or 1 for the causal mask of the forward (key j reaches
 *                    only queries i >= j; lse must come from a causal forward).
 * Errors: FA_ERR_INVALID_ARG (null/misaligned pointers, workspace too small,
 * bad sizes), FA_ERR_UNSUPPORTED (other dtype or d),
 * FA_ERR_CUDA (launch failure).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dO, void* dq, void* dk, void* dv, void* workspace,
           size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
           int dtype, void* stream);

/*
 * Grouped-query backward, the gradient of fa_fwd_gqa: query head h of batch b
 * reads K/V head b*H_kv + h / (H / H_kv), so each K/V head's dK and dV are the
 * sums of the per-query-head gradients over the H / H_kv query heads sharing it
 * (the chain rule through the shared operand; the pages give the forward
 * grouping under "5.4 FlashAttention" and the per-head backward in
 * "FlashAttention-1", 10.2.4).  With H_kv = H this is fa_bwd.
 *
 *   q, o, dO : [B][H][N][d] bfloat16;  lse [B][H][N] float32 (from fa_fwd_gqa).
 *   k, v     : [B][H_kv][N][d] bfloat16.
 *   dq       : [B][H][N][d] bfloat16, written.
 *   dk, dv   : [B][H_kv][N][d] bfloat16, written (the group sums, accumulated
 *              in fp32 on chip and rounded once).
 *   workspace: at least fa_bwd_workspace_size(B, H, N, d) bytes (query heads).
 *   Other arguments as fa_bwd.
 * Errors: as fa_bwd; FA_ERR_INVALID_ARG also for H_kv < 1 or H % H_kv != 0.
 */
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dO, void* dq, void* dk, void* dv, void* workspace,
               size_t workspace_bytes, int B, int H, int H_kv, int N, int d, float scale,
               int causal, int dtype, void* stream);

/*
 * fa_bwd without a caller-supplied workspace, for callers that cannot allocate
 * device memory when they run the backward -- for example a plug-in called
 * from a host framework that owns the device memory budget and forbids
 * allocation inside its execution hook, or a latency-critical caller that
 * cannot afford cudaMalloc's implicit device synchronisation.  The pages have
 * no counterpart to this entry point; it is a deployment convenience.
 *
 * Arguments and results are those of fa_bwd minus (workspace,
 * workspace_bytes).  The scratch is a fixed 64 MiB array inside the library
 * (a file-scope __device__ array that every GPU loading the library holds until
 * the process exits); the call allocates nothing.  Sizes whose
 * fa_bwd_workspace_size() exceeds 64 MiB are refused with FA_ERR_UNSUPPORTED
 * before anything is launched (at d = 64 that allows B*H*ceil128(N) up to
 * 254,200 rows, e.g. B=4, H=16, N=2048).
 *
 * The first call on a device looks up the array's device address for that
 * device (with that device current); make that first call before any stream
 * capture.  All calls on a device share the one array and it keeps the last
 * call's contents: each call writes every scratch region it reads before
 * reading it, so nothing carries over, but calls that overlap in time on the
 * GPU (different streams, or other host threads) race on the array and give
 * wrong results.  FA_ERR_CUDA if the address lookup fails.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, int dtype, void* stream);

/*
 * Synchronise `stream`, then return and clear the current device's status
 * word: FA_OK, or the first device-side error recorded since the last call
 * (FA_ERR_DEVICE_TIMEOUT when a kernel's bounded wait ran out; that kernel
 * returned early and its outputs are undefined).  FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
int fa_last_device_error(void* stream);

/*
 * Upper bound, in nanoseconds of %globaltimer, on any single wait inside a
 * kernel launched after this call on any device (default 2e9 = 2 s; 0 restores
 * the default).  After it runs out the kernel records FA_ERR_DEVICE_TIMEOUT,
 * drains its own in-flight copies and matrix operations (with a fixed 1 s
 * bound), frees its tensor memory and returns.  Tests use a tiny limit to
 * exercise that path; it is not a tuning knob.
 */
void fa_set_wait_timeout_ns(uint64_t ns);

/*
 * Failure-path self test: launch a one-warp kernel whose single wait can never
 * be satisfied (nothing arrives on its barrier).  The bounded wait gives up
 * after the fa_set_wait_timeout_ns() limit and records FA_ERR_DEVICE_TIMEOUT,
 * which the next fa_last_device_error() returns.  Nothing faults or hangs.
 * Returns FA_OK if the kernel was launched.
 */
int fa_selftest_wait_timeout(void* stream);

/* Human-readable name of an fa_status value (static string). */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
