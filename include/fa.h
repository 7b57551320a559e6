/*
 * fa.h -- C ABI of the exact tiled attention library for GB300 (sm_103a).
 *
 * The library computes, for every head of a [B, H, N, d] batch,
 *
 *     scores  = scale * Q K^T            (scale is normally 1/sqrt(d))
 *     weights = row_softmax(scores + mask)
 *     O       = weights V
 *
 * exactly (up to floating-point rounding order), tile by tile with an online
 * softmax, so the N x N score matrix is never written to device memory.
 * Source of the operation: "FlashAttention Interview Questions: IO
 * Complexity, Tiling, and Numerical Stability", section "What is
 * FlashAttention exact about?" (the three-line definition and the statement
 * that the optimisation keeps the mathematical target, mask included), and
 * "FlashAttention 1, 2 & 3: Memory Tiling & Eliminating the O(N^2) HBM
 * Bottleneck", section 1 (Attention(Q,K,V) = softmax(QK^T/sqrt(d))V).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: every tensor is contiguous row-major [B][H][N][d]; the
 *    log-sum-exp and the backward row term are [B][H][N].  One (b, h) pair
 *    is one head; queries and keys have the same length N (the _varlen
 *    calls take separate query and key lengths and per-sequence lengths).
 *  - Types: Q, K, V and dO are bf16 (raw 16-bit storage, `const void*`);
 *    O, LSE, dQ, dK, dV and the workspace are fp32.
 *  - Mask: causal = 0 means no mask; causal = 1 means query i sees key j iff
 *    j <= i.  With this mask no row is ever fully masked.
 *  - Sizes: B, H, N >= 1; d is 64 or 128; B*H*N < 2^31.
 *  - Alignment: Q, K, V, dO, O, dQ, dK, dV must be 16-byte aligned; LSE and
 *    the workspace 4-byte aligned.
 *  - Ownership: every pointer is device memory owned by the caller.  The
 *    library never frees caller memory and never allocates anything whose
 *    size grows with N^2.
 *  - Streams: work is queued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and the calls return before it runs.
 *  - Errors: argument errors are returned synchronously with nothing queued;
 *    launch errors are returned synchronously.  A device-side failure (a
 *    pipeline wait that ran past its time limit) is recorded in a status word
 *    on the device and reported by fa_sync_status().  Every wait inside the
 *    kernels is bounded (4 s by default; the FA_WAIT_LIMIT_MS environment
 *    variable, read once per process, changes it), so a failing kernel
 *    returns instead of hanging.  For tests of that path only,
 *    fa_test_set_stall(n) (initial value: the FA_TEST_STALL_UNIT environment
 *    variable, read once per process) makes the first CTA of every later
 *    launch leave one tile of its n-th work unit unloaded (fa_fwd_decode:
 *    CTA n leaves its first stage unloaded): its waits run out and
 *    fa_sync_status() then reports FA_ERR_TIMEOUT.
 *  - Thread safety: calls may be made from several host threads; calls on
 *    different devices are independent.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same type as cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, causal not 0/1, scale not finite and > 0 */
  FA_ERR_UNSUPPORTED_D = 2, /* d is not 64 or 128 */
  FA_ERR_MISALIGNED = 3,    /* a pointer breaks the alignment rules above */
  FA_ERR_LAUNCH = 4,        /* the CUDA runtime refused a launch or an allocation */
  FA_ERR_TIMEOUT = 5,       /* a kernel wait ran past its limit; the kernel returned early */
  FA_ERR_DEVICE_FAULT = 6   /* the stream reported a CUDA error while synchronising */
} fa_status;

/* Element type of the forward output O (fa_fwd_ex, fa_bwd_ex). */
typedef enum {
  FA_DTYPE_F32 = 0,  /* fp32 O */
  FA_DTYPE_BF16 = 1  /* bf16 O: the fp32 result rounded to nearest even, half the bytes written */
} fa_dtype;

/*
 * Forward pass.
 *   q, k, v : bf16 [B][H][N][d], read only.
 *   o       : fp32 [B][H][N][d], written: O_i = sum_j softmax(s_i)_j v_j.
 *   lse     : fp32 [B][H][N], written: LSE_i = ln sum_j exp(s_ij) over the
 *             eligible keys (natural log of the scaled scores).  This is the
 *             "compact normalization information" the backward pass keeps
 *             ("FlashAttention Interview Questions ...", section "Why can
 *             recomputation help training?").
 *   scale   : multiplier of q.k, finite and > 0 (1/sqrt(d) in the pages'
 *             definition).
 * The online softmax follows the same page, section "How can softmax be
 * computed across tiles?" (running maximum, rescaled sum and accumulator).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_stream_t stream);

/*
 * Forward pass over unequal query/key lengths and padded batches.
 *   q       : bf16 [B][H][Nq][d];  k, v : bf16 [B][H][Nk][d].
 *   o, lse  : fp32 [B][H][Nq][d] and [B][H][Nq].
 *   seqlens_q, seqlens_k : device arrays of B ints, the valid lengths of
 *             each sequence (values clamped to [0, Nq] and [0, Nk]); rows past
 *             them are padding.  NULL means every row is valid.
 * Sequence b uses its first Lq = seqlens_q[b] queries and Lk = seqlens_k[b]
 * keys.  Causal alignment is bottom-right: query i sees key j iff
 * j <= i + (Lk - Lq), so the last query sits at the last key -- the reading
 * of "FlashAttention Interview Questions ...", section "Does subtracting the
 * maximum solve every numerical issue?", which warns that unequal lengths,
 * padding and packed sequences need an explicit alignment.  With Lq = Lk it
 * is the square rule of fa_fwd; a single query (decoding) sees every key.
 * Rows with no eligible key and padding rows are written as O = 0,
 * LSE = -inf.  Padding rows of q, k and v do not affect the result as long as
 * their values are below 1e18 in magnitude (so that every dot product stays
 * finite in fp32).  fa_fwd(...) equals
 * fa_fwd_varlen(..., NULL, NULL, B, H, N, N, ...).  Errors and conventions
 * as fa_fwd; seqlens pointers must be 4-byte aligned.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, float* o, float* lse, const int* seqlens_q,
                        const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                        fa_stream_t stream);

/*
 * Forward pass with each query tile's keys split over several CTAs: the same
 * result as fa_fwd (to fp32 rounding), for batches with too few query tiles
 * to fill the GPU (one head of a few thousand tokens has a few dozen).  Each
 * split runs the online softmax ("FlashAttention Interview Questions ...",
 * section "How can softmax be computed across tiles?") over its own range of
 * key tiles and leaves a normalised partial output and its log-sum-exp; a
 * second kernel merges the partials by that log-sum-exp -- the same
 * merge-by-rescaling the online softmax applies from tile to tile.  The
 * library picks the number of splits from the device's SM count (at most
 * 16, at least two key tiles each); when one split suffices it runs fa_fwd.
 *   workspace : fp32 scratch of fa_fwd_splitkv_workspace_bytes(B, H, N, d)
 *               bytes, 16-byte aligned; or NULL (a stream-ordered allocation,
 *               freed on the same stream).
 * Other arguments, results and errors as fa_fwd.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, float* o, float* lse, float* workspace, int B,
                         int H, int N, int d, float scale, int causal, fa_stream_t stream);

/* Bytes of the fa_fwd_splitkv workspace (an upper bound that does not depend
 * on the device); 0 on invalid sizes. */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int d);

/* Most query rows per head that fa_fwd_decode accepts. */
#define FA_DECODE_MAX_Q 8

/*
 * The general forward: fa_fwd_varlen with a choice of output type.
 *   o       : [B][H][Nq][d] of o_dtype (FA_DTYPE_F32 or FA_DTYPE_BF16),
 *             16-byte aligned.  With FA_DTYPE_BF16 each element is the fp32
 *             result of fa_fwd_varlen rounded to the nearest bf16 (ties to
 *             even); LSE stays fp32.
 * Other arguments, results and errors as fa_fwd_varlen; an o_dtype outside
 * the enum returns FA_ERR_INVALID_ARG.  fa_fwd_varlen(...) equals
 * fa_fwd_ex(..., FA_DTYPE_F32, ...).
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, int o_dtype, float* lse,
                    const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                    int causal, fa_stream_t stream);

/*
 * Forward pass with a general additive mask: the "+ mask" of the definition
 * weights = row_softmax(scores + mask) ("FlashAttention Interview Questions
 * ...", section "What is FlashAttention exact about?") as a bias added to
 * the scaled scores, s_ij = scale * q_i.k_j + bias_ij.  It is not scaled; an
 * entry of -inf hides the key; it combines with the causal rule and with
 * padding, and a row whose keys are all hidden gets O = 0, LSE = -inf.
 *   bias  : bf16, element (b, h, i, j) at
 *           bias + b*bias_stride_b + h*bias_stride_h + i*bias_stride_q + j,
 *           keys contiguous.  Strides in elements, >= 0; 0 broadcasts over
 *           that index (bias_stride_q = 0: one row of key biases for every
 *           query, e.g. a key-padding mask); otherwise bias_stride_q >= Nk.
 *           2-byte aligned.  Rows that start on a 16-byte boundary (base
 *           16-byte aligned, strides multiples of 8) are read in 16-byte
 *           loads, others element by element (slower).  No +inf, no NaN.
 * Other arguments, results and errors as fa_fwd_ex; a null bias or an
 * invalid stride returns FA_ERR_INVALID_ARG, a bias at an odd address
 * FA_ERR_MISALIGNED.  Gradients of a masked forward: fa_bwd_bias.
 */
fa_status fa_fwd_bias(const void* q, const void* k, const void* v, void* o, int o_dtype, float* lse,
                      const void* bias, long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                      const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, fa_stream_t stream);

/*
 * FP8 forward: fa_fwd with E4M3 inputs ("FlashAttention 1, 2 & 3", section on
 * FlashAttention-3: FP8 on the tensor cores).  q8, k8: [B][H][N][128] E4M3
 * (one byte each); vt8: V transposed, [B][H][128][N] E4M3; o fp32
 * [B][H][N][128], lse fp32 [B][H][N], as fa_fwd.  Scores and both products
 * accumulate in fp32 from the E4M3 values as given (descale factors of q and
 * k fold into `scale`; one of v multiplies O, which the caller applies);
 * the probabilities P are rounded to E4M3 before O = P V, so O carries an
 * error of up to 2^-4 sum_j P_ij |v_j| plus a subnormal term against the
 * exact result on the same inputs; LSE does not (it sums the unrounded P).
 * d must be 128 (else FA_ERR_UNSUPPORTED_D); N a multiple of 16 (rows of
 * vt8 are whole 16-byte groups; else FA_ERR_INVALID_ARG); square sequences,
 * causal or not.  All pointers 16-byte aligned (lse 4).  Errors and
 * asynchrony as fa_fwd.
 */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, float* o, float* lse, int B, int H, int N,
                     int d, float scale, int causal, fa_stream_t stream);

/*
 * Decode-shaped forward: 1 <= Nq <= FA_DECODE_MAX_Q query rows per head
 * against a long key/value history.  Computes exactly what fa_fwd_varlen
 * computes for the same arguments (same layouts, lengths, bottom-right causal
 * alignment, padding rules and outputs), with a kernel built for this shape:
 * single-token decoding reads all of K and V once per step for one query row,
 * about one FLOP per byte, so it is bound by HBM bandwidth rather than by the
 * tensor cores ("FlashAttention Interview Questions ...", final section, on
 * prefill against single-token decoding).  Each head's keys are split over
 * many CTAs that stream K/V once; a second kernel merges the splits by their
 * log-sum-exp.
 *   workspace : fp32 scratch for the per-split results,
 *               fa_fwd_decode_workspace_bytes(B, H, Nq, Nk, d) bytes,
 *               16-byte aligned; or NULL, in which case the library takes a
 *               stream-ordered allocation when it splits the keys and frees
 *               it on the same stream.
 * Errors as fa_fwd_varlen; Nq outside [1, FA_DECODE_MAX_Q] returns
 * FA_ERR_INVALID_ARG.
 */
fa_status fa_fwd_decode(const void* q, const void* k, const void* v, float* o, float* lse, const int* seqlens_q,
                        const int* seqlens_k, float* workspace, int B, int H, int Nq, int Nk, int d, float scale,
                        int causal, fa_stream_t stream);

/* Bytes of the fa_fwd_decode workspace (an upper bound that does not depend
 * on the device); 0 on invalid sizes. */
size_t fa_fwd_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/*
 * Backward pass by recomputation: attention probabilities are rebuilt from
 * q, k and the saved lse instead of being stored ("FlashAttention Interview
 * Questions ...", section "Why can recomputation help training?").
 *   q, k, v, dO : bf16 [B][H][N][d], read only (dO = dL/dO).
 *   o, lse      : fp32 outputs of fa_fwd for the same q, k, v, scale, causal.
 *   dq, dk, dv  : fp32 [B][H][N][d], overwritten with dL/dQ, dL/dK, dL/dV.
 *   workspace   : fp32 buffer of fa_bwd_workspace_bytes(B, H, N) bytes that
 *                 receives the row term D_i = sum_j P_ij dP_ij (formed from
 *                 rowsum(dO o O) and corrected to the probabilities the
 *                 backward pass recomputes); or NULL, in which case the
 *                 library takes a stream-ordered allocation and frees it on
 *                 the same stream.
 * Computes P_ij = exp(s_ij - LSE_i), dV = P^T dO, dP = dO V^T,
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse, const void* dO,
                 float* dq, float* dk, float* dv, float* workspace, int B, int H, int N, int d, float scale,
                 int causal, fa_stream_t stream);

/*
 * Backward pass over unequal query/key lengths and padded batches, the
 * gradient of fa_fwd_varlen for the same arguments.
 *   q, dO, o    : [B][H][Nq][d] (q, dO bf16; o fp32);  lse : fp32 [B][H][Nq].
 *   k, v        : bf16 [B][H][Nk][d].
 *   dq          : fp32 [B][H][Nq][d];  dk, dv : fp32 [B][H][Nk][d], overwritten.
 *   workspace   : fp32, fa_bwd_workspace_bytes(B, H, Nq) bytes, or NULL as
 *                 for fa_bwd; it ends holding D for each query row.
 *   seqlens_q, seqlens_k : as fa_fwd_varlen (NULL: every row valid).
 * Alignment and masking follow fa_fwd_varlen.  Padding rows and rows with no
 * eligible key get zero gradients (and D = 0); key rows past the valid length
 * get dK = dV = 0.  Padding rows of q, k, v and dO do not affect the result
 * under the same bound as fa_fwd_varlen.  fa_bwd(...) equals
 * fa_bwd_varlen(..., NULL, NULL, B, H, N, N, ...).
 */
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const float* o, const float* lse,
                        const void* dO, float* dq, float* dk, float* dv, float* workspace, const int* seqlens_q,
                        const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                        fa_stream_t stream);

/*
 * The general backward: fa_bwd_varlen taking O of either output type of
 * fa_fwd_ex (o_dtype as there).  O only enters through the row term
 * D_i = sum_c dO_ic O_ic, which the dQ stage corrects to the exact
 * sum_j P_ij dP_ij of the recomputed probabilities, so a bf16 O leaves the
 * gradients' accuracy unchanged.  fa_bwd_varlen(...) equals
 * fa_bwd_ex(..., FA_DTYPE_F32, ...).
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, int o_dtype, const float* lse,
                    const void* dO, float* dq, float* dk, float* dv, float* workspace, const int* seqlens_q,
                    const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    fa_stream_t stream);

/* Gradients of fa_fwd_bias ("FlashAttention Interview Questions", sections
 * "What is FlashAttention exact about?" for the mask and "Why can
 * recomputation help training?" for the backward from the saved LSE):
 * fa_bwd_ex with the same additive mask (bias and its strides exactly as
 * passed to the forward call that made o and lse).
 * The mask enters only the recomputed probabilities,
 * P_ij = exp(scale * q_i.k_j + bias_ij - LSE_i); it is a constant of the
 * differentiation, so no gradient of the mask is formed.  Rows whose keys
 * the mask hides entirely (LSE = -inf) get dQ = 0 and add nothing to dK, dV.
 * Mask rows that start on a 16-byte boundary are read in 16-byte loads by the
 * dQ kernel; the dK/dV kernel reads the mask down its columns, one 2-byte
 * load per (query, key) per pass, coalesced over 32 consecutive keys.
 * Errors as fa_bwd_ex and fa_fwd_bias. */
fa_status fa_bwd_bias(const void* q, const void* k, const void* v, const void* o, int o_dtype, const float* lse,
                      const void* dO, const void* bias, long long bias_stride_b, long long bias_stride_h,
                      long long bias_stride_q, float* dq, float* dk, float* dv, float* workspace,
                      const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale,
                      int causal, fa_stream_t stream);

/*
 * Largest B*H*N that fa_bwd_noalloc accepts: 2^20 rows, i.e. 4 MiB of fp32
 * scratch held in a static device array by every GPU that loads the library,
 * for as long as the library stays loaded.
 */
#define FA_NOALLOC_MAX_ROWS (1 << 20)

/*
 * fa_bwd without any allocation.  The pages describe no such call: it exists
 * for callers that cannot allocate device memory when they run the backward
 * pass -- a host framework or inference runtime that owns every byte of
 * device memory through its own pool and forbids libraries to allocate behind
 * its back, or a latency-critical loop that reserved all memory up front and
 * must not risk an allocation (or an out-of-memory failure) on its hot path.
 *
 * Arguments and results are those of fa_bwd, minus the workspace: the row
 * term D lives in a fixed device array inside the library (see
 * FA_NOALLOC_MAX_ROWS).  The call makes no cudaMalloc/cudaFree or other
 * allocating call.  Its first call on a device looks up that array's device
 * address (cudaGetSymbolAddress) with the caller's device current; make that
 * first call before any stream capture on the device.
 *
 * Errors: as fa_bwd; B*H*N above FA_NOALLOC_MAX_ROWS returns
 * FA_ERR_INVALID_ARG with nothing queued.  All calls on one device share the
 * array, and it keeps the last call's contents (every call rewrites all of
 * the rows it uses before reading them): two calls whose work overlaps on the
 * GPU (different streams, not ordered) race on it and give wrong gradients.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const float* o, const float* lse,
                         const void* dO, float* dq, float* dk, float* dv, int B, int H, int N, int d, float scale,
                         int causal, fa_stream_t stream);

/*
 * Single-pass backward: the same gradients as fa_bwd_bias (bias NULL: as
 * fa_bwd_varlen), with dQ formed inside the dK/dV sweep instead of by a
 * second sweep that recomputes S and dP ("FlashAttention Interview Questions
 * ...", section "Why can recomputation help training?": P is rebuilt from
 * q, k and the saved lse).  Two kernels run in stream order:
 *   1. the row term D_i = sum_j P_ij dP_ij, formed from the recomputed fp32
 *      probabilities (two tensor-core products per tile, S = q k^T and
 *      dP = dO v^T); it also sets dQ to zero;
 *   2. one CTA per 128-key tile sweeps the query tiles that see it and forms
 *      dV += P^T dO, dK += scale dS^T q and each tile's dQ share
 *      scale dS k, which it adds into dQ in place.
 * The row term comes from P and dP, not from the forward output, so no O is
 * taken.  dQ's sum over key tiles runs in an order that varies between runs,
 * so dQ may differ in its last bits from call to call (dK, dV do not).
 *   q, k, v, dO, lse, dq, dk, dv, seqlens_q, seqlens_k, B, H, Nq, Nk, d,
 *   scale, causal : as fa_bwd_varlen.
 *   bias and its strides : as fa_bwd_bias, or bias = NULL for no mask.
 *   workspace : fp32, fa_bwd_workspace_bytes(B, H, Nq) bytes, ends holding D;
 *               or NULL (a stream-ordered allocation, freed on the stream).
 * Errors as fa_bwd_bias.
 */
fa_status fa_bwd_single_pass(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                             const void* bias, long long bias_stride_b, long long bias_stride_h,
                             long long bias_stride_q, float* dq, float* dk, float* dv, float* workspace,
                             const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq, int Nk, int d,
                             float scale, int causal, fa_stream_t stream);

/*
 * One stage of a backward pass, for callers that time or schedule the
 * kernels separately; the workspace is required (never NULL).
 *   stage 0: dQ; also writes the exact row term D_i = sum_j P_ij dP_ij into
 *            the workspace (formed from rowsum(dO o O) inside the kernel).
 *   stage 1: dK and dV (needs stage 0 first).
 *            Stages 0, 1 in order on one stream are exactly fa_bwd.
 *   stage 2: the row term D from the recomputed P and dP, and dQ = 0
 *            (o is not read and may be NULL).
 *   stage 3: dK, dV, and dQ accumulated into place (needs stage 2 first).
 *            Stages 2, 3 in order are fa_bwd_single_pass without a mask.
 * Arguments as fa_bwd; a stage outside 0..3 returns FA_ERR_INVALID_ARG.
 */
fa_status fa_bwd_stage(int stage, const void* q, const void* k, const void* v, const float* o, const float* lse,
                       const void* dO, float* dq, float* dk, float* dv, float* workspace, int B, int H, int N, int d,
                       float scale, int causal, fa_stream_t stream);

/* Bytes of the fa_bwd workspace: B*H*N fp32 values (0 on invalid sizes);
 * for fa_bwd_varlen pass N = Nq. */
size_t fa_bwd_workspace_bytes(int B, int H, int N);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns FA_ERR_DEVICE_FAULT if the stream reported a CUDA
 * error, FA_ERR_TIMEOUT if a kernel wait ran out since the last call, FA_OK
 * otherwise.
 */
fa_status fa_sync_status(fa_stream_t stream);

/*
 * Details of the last device-side failure read by fa_sync_status():
 * out[0] status code, out[1] wait site, out[2] block index, out[3] work unit.
 * Wait sites: 1-7 forward, 11-20 dK/dV, 21-32 dQ, 35-36 decode, 41-47 FP8
 * forward, 51-59 the single-pass row-term pass, 61-63 the single-pass dK/dV
 * sweep (each kernel's source names them).
 * Returns FA_OK, or FA_ERR_INVALID_ARG if out is NULL.
 */
fa_status fa_last_failure(int out[4]);

/*
 * Testing hook of the timeout path (see "Errors" above): from the next call
 * on, the first CTA of each launch leaves one tile of its unit-th work unit
 * unloaded, so that the waits on it run out and fa_sync_status() reports
 * FA_ERR_TIMEOUT; unit = -1 switches the hook off (the default unless
 * FA_TEST_STALL_UNIT was set when the library first launched work).  Nothing
 * faults or hangs.  Returns FA_OK, or FA_ERR_INVALID_ARG for unit < -1.
 */
fa_status fa_test_set_stall(int unit);

/* Static, human-readable name of a status code; never NULL. */
const char* fa_status_string(fa_status s);

/*
 * Host-only view of the persistent scheduler, for tests and tools (no GPU
 * needed).  Deals the ceil(N/256) two-tile work units of each of `heads`
 * heads to `grid` CTAs exactly as the forward kernel does.  Writes up to
 * `capacity` triples (cta, head, pair) in dealing order and returns how many
 * units exist in total, or -1 on invalid arguments.  l2_budget_bytes sets how
 * many heads share an L2 group (0 = the library default).
 */
long long fa_sched_enumerate(int heads, int N, int d, int causal, int grid, long long l2_budget_bytes,
                             int* out_cta, int* out_head, int* out_pair, long long capacity);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
