/*
 * sdpa.h -- C ABI of the GB300 (sm_103a) exact scaled dot-product attention.
 *
 * The operation (SDPA tutorial page "(Beta) Implementing High-Performance
 * Transformers with Scaled Dot Product Attention", section "Overview"):
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 *
 * computed IO-aware as in the FlashAttention news article (QbitAI repost,
 * section "FlashAttention"): the kernels tile Q and K/V through on-chip
 * memory so the Lq x Lk score matrix never reaches HBM; the forward keeps a
 * running row maximum and row sum across K/V blocks and saves the per-row
 * log-sum-exp, and the backward recomputes the probabilities from Q, K and
 * that log-sum-exp instead of storing them.
 *
 * General rules for every call:
 *  - All tensor arguments are DEVICE pointers owned by the caller, on the
 *    device that is current for the calling thread. The library allocates
 *    nothing, keeps no reference after the call returns, and runs
 *    asynchronously on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Tensors are contiguous (except in the *_strided calls). Element type is
 *    `dtype` (sdpa_dtype) for q/k/v/o/dO/dq/dk/dv; lse is always float32.
 *  - Dense layout (cu_seqlens == NULL): q, o, dO, dq are [B, H, Lq, d];
 *    k, v, dk, dv are [B, H, Lk, d]; lse is [B, H, Lq].
 *  - Packed variable-length layout (cu_seqlens != NULL; the tutorial's
 *    NestedTensor batches, section "NestedTensor and Dense tensor support"):
 *    q, k, v, o (and gradients) are [total, H, d] with the tokens of
 *    sequence s at rows cu_seqlens[s] .. cu_seqlens[s+1]-1; the same offsets
 *    serve queries and keys (self-attention). `cu_seqlens` is a device int32
 *    array of B+1 non-decreasing offsets starting at 0. In this mode B is the
 *    number of sequences, Lq is the packed token count `total`
 *    (= cu_seqlens[B]) and Lk is an upper bound on every sequence length
 *    (max_seqlen); lse is [H, total].
 *  - Causal masking is top-left aligned: query i sees keys j <= i (within its
 *    sequence when packed).
 *  - Return value: SDPA_OK or a negative sdpa_status. Argument errors are
 *    detected on the host before anything is launched. A nonzero return
 *    leaves a message for sdpa_last_error(). Errors found by a kernel while
 *    it runs (a bounded wait that gave up, a packed sequence longer than its
 *    bound) are recorded in a device status word that sdpa_device_status()
 *    reads.
 *  - Packed cross-attention (sdpa_fwd_varlen / sdpa_bwd_varlen): queries and
 *    keys of sequence s sit on two different token axes, q/o/dO/dq
 *    [total_q, H, d] at rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 and
 *    k/v/dk/dv [total_k, H, d] at rows cu_seqlens_k[s] .. cu_seqlens_k[s+1]-1;
 *    lse is [H, total_q]. Query i of a sequence attends to the keys of the
 *    same sequence (causal: to its keys j <= i). The same calls cover a
 *    padded-free [B, L, H, d] batch: pass the uniform offsets s*L.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SDPA_F32 = 0, SDPA_F16 = 1, SDPA_BF16 = 2 } sdpa_dtype;

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_ARG = -1,         /* null pointer, non-positive size, bad scale, Lk = 0 with Lq > 0 */
  SDPA_ERR_UNSUPPORTED = -2, /* head dim / dtype / mode this build does not implement */
  SDPA_ERR_CUDA = -3,        /* a CUDA runtime call failed (message names it) */
  SDPA_ERR_TIMEOUT = -4,     /* a kernel's bounded wait gave up (from sdpa_device_status) */
  SDPA_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than sdpa_bwd_workspace_size() */
  SDPA_ERR_BOUNDS = -6       /* debug build: a device-side bounds check failed (from sdpa_device_status) */
} sdpa_status;

/* Bits of the device status word (see sdpa_device_status). */
#define SDPA_STATUS_TIMEOUT 1u   /* an mbarrier wait exceeded its time limit; outputs invalid */
#define SDPA_STATUS_SEQLEN 2u    /* a packed sequence is longer than its bound (max_seqlen), or has
                                    queries but no keys; its outputs are left unwritten */
#define SDPA_STATUS_BOUNDS 4u    /* debug build only: a device-side bounds check failed and the
                                    access it guarded was skipped; outputs invalid */

/*
 * Forward: O and LSE.
 *   q, k, v : inputs (layouts above), dtype `dtype`.
 *   o       : output, same layout as q.
 *   lse     : float32 output, natural-log log-sum-exp of each query row
 *             (lse_i = log sum_j exp(scale * q_i . k_j) over visible j).
 *   B, H, Lq, Lk, d : sizes (packed mode: see the layout rules above).
 *   scale   : the softmax scale (usually 1/sqrt(d)); must be finite.
 *   is_causal : 0 or 1.
 * Supported: dtype F32 with d <= 128 (plain fp32 arithmetic, no TF32);
 * F16 / BF16 with d in {32, 64, 128} (tensor cores, fp32 accumulation).
 * Lq == 0 (or B == 0 / H == 0) is a no-op that returns SDPA_OK.
 */
int sdpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
             const int* cu_seqlens, int dtype, void* stream);

/*
 * Forward over packed sequences whose queries and keys have their own
 * offsets (cross-attention over a NestedTensor-style batch; layout rules
 * above). The tutorial's NestedTensor section runs the op on batches of
 * unequal lengths; this is that op with the key side indexed separately.
 *   nseq          : number of sequences; cu_seqlens_q / cu_seqlens_k are
 *                   device int32 arrays of nseq+1 non-decreasing offsets
 *                   from 0 to total_q / total_k.
 *   max_seqlen_q, max_seqlen_k : upper bounds on every sequence's query and
 *                   key length (sizes the launch; a longer sequence sets
 *                   SDPA_STATUS_SEQLEN and is left unwritten).
 *   o, lse        : [total_q, H, d] and [H, total_q] outputs.
 * A sequence with queries must have at least one key (else
 * SDPA_STATUS_SEQLEN); total_q == 0 or max_seqlen_q == 0 is a no-op;
 * max_seqlen_k == 0 or total_k == 0 with queries present is SDPA_ERR_ARG.
 * dtype / d support as for sdpa_fwd.
 */
int sdpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    int nseq, int H, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                    int d, float scale, int is_causal,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int dtype, void* stream);

/*
 * Forward over dense tensors at any element strides: the SDPA tutorial's
 * module (section "Causal Self Attention") projects to [B, L, H * d] and
 * views it as [B, L, H, d].transpose(1, 2), a [B, H, L, d] tensor whose rows
 * are H * d elements apart; this call reads and writes such views in place,
 * with no copy.
 *   strides : HOST array of 12 element strides, (batch, head, row) for q, k,
 *             v and o in that order; the head dim is contiguous (stride 1).
 *             A dimension longer than 1 needs a positive stride; fp16 / bf16
 *             strides must be multiples of 8 elements (16 bytes) and the
 *             bases 16-byte aligned. Rows of o must not overlap.
 *   lse     : contiguous [B, H, Lq] float32, as for sdpa_fwd.
 * Other arguments, support and errors as for sdpa_fwd with cu_seqlens = NULL.
 */
int sdpa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                     const long long* strides, int dtype, void* stream);

/*
 * Bytes of device workspace sdpa_bwd needs for these sizes (a float32 row
 * statistic D = rowsum(dO * O) and a float32 dQ accumulator, both over the
 * query rows). The FlashAttention news article (QbitAI repost, section
 * "FlashAttention") has the backward rebuild the attention matrix from the
 * inputs instead of storing it; these two arrays, linear in the query rows,
 * are what that rebuild keeps between its kernels. Packed mode: pass B = 1
 * and Lq = total. Never fails; returns 0 when nothing is needed.
 */
size_t sdpa_bwd_workspace_size(int B, int H, int Lq, int d, int dtype);

/*
 * Backward: gradients of sum(dO * O) w.r.t. q, k, v. As the FlashAttention
 * news article (QbitAI repost, section "FlashAttention") describes, the
 * probabilities are not stored by the forward but rebuilt here from q, k and
 * the forward's lse.
 *   q, k, v, o, lse : the forward's inputs and outputs (o and lse exactly as
 *                     sdpa_fwd wrote them).
 *   dO      : upstream gradient, layout of o.
 *   dq, dk, dv : outputs, layouts of q, k, v; fully overwritten.
 *   workspace : device scratch of at least sdpa_bwd_workspace_size() bytes,
 *               256-byte aligned; its contents on entry do not matter.
 * Other arguments as for sdpa_fwd, dense or packed (cu_seqlens != NULL; the
 * workspace is then sized with B = 1 and Lq = total). Supported: F32 with
 * d <= 128; F16/BF16 with d in {32, 64, 128}.
 */
int sdpa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv,
             int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
             const int* cu_seqlens, int dtype,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward over dense tensors at any element strides (the backward of
 * sdpa_fwd_strided).
 *   strides : HOST array of 24 element strides, (batch, head, row) for q, k,
 *             v, o, dO, dq, dk and dv in that order; rules as for
 *             sdpa_fwd_strided. lse contiguous; the workspace as for sdpa_bwd
 *             (its fp32 dQ accumulator is contiguous whatever dq's strides).
 * Other arguments, support and errors as for sdpa_bwd with cu_seqlens = NULL.
 */
int sdpa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv,
                     int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                     const long long* strides, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward of sdpa_fwd_varlen: dq [total_q, H, d], dk and dv [total_k, H, d],
 * fully overwritten. Arguments as for sdpa_fwd_varlen plus those of sdpa_bwd;
 * the workspace is sdpa_bwd_workspace_size(1, H, total_q, d, dtype) bytes.
 * Supported: F32 with d <= 128; F16/BF16 with d in {32, 64, 128}.
 */
int sdpa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv,
                    int nseq, int H, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                    int d, float scale, int is_causal,
                    const int* cu_seqlens_q, const int* cu_seqlens_k, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-sparse attention (the FlashAttention news article, QbitAI repost,
 * section "FlashAttention", names "block-sparse FlashAttention" without
 * defining it): exact attention restricted to the score tiles that a 0/1
 * block mask keeps, with every other score excluded like a causally masked
 * one; the kernels skip the dropped tiles. Dense layout only.
 *   block_mask : device uint8 array; tile (qb, kb) of head (b, h), covering
 *                query rows [128 qb, 128 qb + 128) and keys [128 kb, 128 kb + 128),
 *                is kept iff block_mask[b * mask_stride_b + h * mask_stride_h
 *                + qb * mask_stride_row + kb] != 0, for qb < ceil(Lq / 128),
 *                kb < ceil(Lk / 128). Strides are in elements; 0 broadcasts a
 *                mask over the batch or the heads; mask_stride_row must be at
 *                least ceil(Lk / 128).
 *   A query row with no visible key (all its tiles dropped, or dropped and
 *   causally masked) gets O = 0 and LSE = -inf, and no gradient.
 * Other arguments, support and errors as for sdpa_fwd with cu_seqlens = NULL.
 */
int sdpa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                         const unsigned char* block_mask, long long mask_stride_b,
                         long long mask_stride_h, int mask_stride_row, int dtype, void* stream);

/*
 * Backward of sdpa_fwd_blocksparse (same mask; o and lse as that call wrote
 * them). Arguments, workspace and support as for sdpa_bwd with
 * cu_seqlens = NULL; Lq is limited to 131072 (SDPA_ERR_UNSUPPORTED above).
 */
int sdpa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv,
                         int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                         const unsigned char* block_mask, long long mask_stride_b,
                         long long mask_stride_h, int mask_stride_row, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Attention with an additive mask (the SDPA tutorial's attn_mask argument,
 * section "Causal Self Attention"): O = softmax(scale * Q K^T + M) V, with
 * the causal mask on top when is_causal = 1. Dense layout only.
 *   attn_mask : device array in the input dtype; M(b, h, i, j) =
 *               attn_mask[b * mask_stride_b + h * mask_stride_h
 *               + i * mask_stride_row + j] for i < Lq, j < Lk (keys
 *               contiguous). Strides are in elements; 0 broadcasts over the
 *               batch or the heads. Entries are finite or -inf (-inf excludes
 *               the score). fp16/bf16: the base must be 16-byte aligned and
 *               the strides multiples of 8 elements (the tensor-core kernels
 *               read the mask with TMA), so mask_stride_row is at least Lk
 *               rounded up to 8; entries past Lk are never read. fp32: row
 *               stride at least Lk.
 *   A query row with no visible key gets O = 0 and LSE = -inf, and no gradient.
 * LSE is the log-sum-exp of the masked scores. Other arguments, support and
 * errors as for sdpa_fwd with cu_seqlens = NULL.
 */
int sdpa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                    const void* attn_mask, long long mask_stride_b, long long mask_stride_h,
                    long long mask_stride_row, int dtype, void* stream);

/*
 * Backward of sdpa_fwd_masked (same mask; o and lse as that call wrote them).
 * Gradients for q, k and v only (none for the mask). Arguments, workspace and
 * support as for sdpa_bwd with cu_seqlens = NULL.
 */
int sdpa_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv,
                    int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                    const void* attn_mask, long long mask_stride_b, long long mask_stride_h,
                    long long mask_stride_row, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Attention with dropout on the probabilities (the SDPA tutorial's
 * dropout_p argument, section "Causal Self Attention"):
 * O = (P * Z) V with P = softmax(scale * Q K^T [+ causal mask]) and Z = 0
 * for a dropped score, 1/(1 - p') for a kept one; LSE is that of the full
 * softmax. Dense layout only.
 *   dropout_p : in [0, 1); used as p' = t / 256 with t = round(256 p)
 *               (t = 0 is no dropout).
 *   seed      : 64-bit key of the generator. Score (i, j) of head
 *               u = b * H + h is kept iff byte (j mod 16) (little-endian
 *               within the 32-bit words) of Philox4x32-10 (Salmon et al.,
 *               SC 2011) at counter (j / 16, i, u, 0) and key
 *               (seed mod 2^32, seed / 2^32) is at least t.
 * Other arguments, support and errors as for sdpa_fwd with cu_seqlens = NULL.
 */
int sdpa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                     float dropout_p, unsigned long long seed, int dtype, void* stream);

/*
 * Backward of sdpa_fwd_dropout: the same dropout_p and seed reproduce the
 * forward's keep pattern. Arguments, workspace and support as for sdpa_bwd
 * with cu_seqlens = NULL.
 */
int sdpa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv,
                     int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                     float dropout_p, unsigned long long seed, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass for callers that cannot allocate device memory: it takes the
 * same arguments as sdpa_bwd except the workspace and cu_seqlens (dense
 * layout only), and uses a scratch array of 16 MiB compiled into the library
 * instead. The pages have no counterpart to this call; it exists because some
 * callers run where no allocation is possible -- a pre-sized memory pool that
 * must not grow, a plugin or embedded runtime that is handed only its input
 * and output buffers, a host that forbids cudaMalloc after start-up.
 *   Limit: sdpa_bwd_workspace_size(B, H, Lq, d, dtype) must not exceed
 *   16 MiB (B*H*Lq*(d+1)*4 bytes, rounded, for fp16/bf16); larger problems
 *   return SDPA_ERR_WORKSPACE before anything is launched.
 *   The first call on each device looks up the array's device address while
 *   that device is current. With CUDA's lazy module loading (the default)
 *   that lookup is also what loads the array onto the device and reserves
 *   its 16 MiB, so a caller with a fixed memory budget should make the first
 *   call at start-up, and before any stream capture. Later calls on that
 *   device allocate nothing.
 *   Every call on a device shares the one array (it is held until the process
 *   exits and keeps the last call's contents; each call re-initialises what it
 *   needs), so calls whose kernels may overlap on the GPU race and must be
 *   ordered by the caller (same stream, or events).
 */
int sdpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv,
                     int B, int H, int Lq, int Lk, int d, float scale, int is_causal,
                     int dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device. Returns SDPA_OK, SDPA_ERR_TIMEOUT (bit SDPA_STATUS_TIMEOUT
 * was set), SDPA_ERR_BOUNDS (bit SDPA_STATUS_BOUNDS, debug build), SDPA_ERR_ARG
 * (bit SDPA_STATUS_SEQLEN was set) or SDPA_ERR_CUDA.
 * If `bits` is not NULL the raw word is stored there.
 */
int sdpa_device_status(void* stream, unsigned* bits);

/*
 * Kernel timing aid (no counterpart on the pages: it serves measurement).
 * Installs two CUDA events (cudaEvent_t handles the caller created, with
 * timing enabled) that every later call records on its own stream directly
 * before and directly after its main attention kernel: the tensor-core (or
 * fp32) forward kernel for which = 0, the backward's for which = 1 (the
 * backward's row-statistic pass and dQ conversion fall outside the pair).
 * cudaEventElapsedTime on the pair then gives the last such kernel's device
 * time. NULL for both removes them. The setting is process-wide and not
 * synchronised: install events from one thread, with no calls in flight on
 * other threads. Returns SDPA_OK, or SDPA_ERR_ARG for another `which` or a
 * single NULL.
 */
int sdpa_trace_events(int which, void* begin_event, void* end_event);

/*
 * Testing aid: sets debug flags for later calls on any thread and returns the
 * previous value. Flag 1 makes the forward tensor-core kernel skip its Q load,
 * so every wait in it runs out and sdpa_device_status() reports
 * SDPA_ERR_TIMEOUT after about a second. Flag 2 (debug build only) makes the
 * forward's bounds checks take O as one row shorter than it is, so the store
 * of its last row is refused and skipped and sdpa_device_status() reports
 * SDPA_ERR_BOUNDS. 0 (the default) is normal operation.
 */
int sdpa_debug_set(int flags);

/*
 * 1 for the debug build (compiled with SDPA_DEBUG: device-side bounds checks
 * on the kernels' stores, reductions and shared-memory staging; a failed
 * check skips the access and sets SDPA_STATUS_BOUNDS, nothing traps), 0 for
 * the normal build, whose kernels carry no checks.
 */
int sdpa_debug_build(void);

/*
 * Message for the last nonzero return on the calling thread ("" if none).
 * The SDPA tutorial's calls raise RuntimeError with a message when an input
 * is not supported (section "Explicit Dispatcher Control"); the Python
 * binding raises with this text.
 */
const char* sdpa_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int sdpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
