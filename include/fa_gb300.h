/*
 * fa_gb300.h -- exact scaled-dot-product attention forward on GB300 (sm_103a).
 *
 * Operation (FlashAttention from Scratch, sec. 2 "Begin with one attention
 * row"; FlashAttention Cheat Sheet, sec. 1 "The whole operation"):
 *
 *     O = softmax(Q K^T * softmax_scale + M) V,   LSE_i = ln sum_j exp(s_ij)
 *
 * computed tile by tile with the online-softmax recurrence (running maximum,
 * running sum, unnormalised accumulator; Cheat Sheet sec. 5) so that the
 * score matrix never reaches device memory.  M is 0 for allowed pairs and
 * -inf otherwise.  With causal != 0 key j is allowed for query i iff
 * j <= i + (Lk - Lq): the queries are the last Lq positions of the key
 * sequence (bottom-right alignment; FlashAttention from Scratch, sec. 5
 * "Rectangular causal masking is a correctness issue").  A query row with no
 * allowed key gets O = 0 and LSE = -inf (sec. 4.4 "Handle the empty state
 * deliberately").  LSE is in natural-log units (sec. 6.3).
 *
 * Grouped-query attention: Hq must be a multiple of Hkv and query head h
 * reads KV head h / (Hq / Hkv) (sec. 9.2 "GQA and MQA change decode
 * traffic"); K and V are not replicated.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers on the current CUDA device, 16-byte
 *    aligned, and owned by the caller.  Q, K, V are read only; O and LSE are
 *    fully overwritten (including fully masked rows and rows of empty
 *    sequences).  Output buffers must not overlap the inputs.
 *  - Q, K, V are bf16 (raw 16-bit storage, passed as void*).  O and LSE are
 *    fp32: the kernel accumulates in fp32, and a bf16 O could not honour an
 *    absolute error of 1e-2 once |O| >= 4 (half a bf16 ulp is 1/64 there).
 *  - Head dimension D must be 64 or 128.
 *  - The call is asynchronous on `stream` (0 = legacy default stream) and
 *    never synchronises it.  Errors detected inside a kernel (a pipeline wait
 *    that exceeded its time limit) are latched on the device and reported by
 *    the next fa_check().
 *  - Nothing throws across this interface: every call returns a status.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <cuda_runtime_api.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, Hq % Hkv != 0,
                               non-finite or non-positive scale, misalignment */
    FA_ERR_UNSUPPORTED = 2, /* D not in {64, 128}, or no sm_103 device */
    FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed */
    FA_ERR_TIMEOUT = 4      /* a kernel pipeline wait hit its time limit */
} fa_status_t;

/*
 * Dense batched attention forward.
 *
 *   q   [B, Hq,  Lq, D] bf16, contiguous row-major
 *   k   [B, Hkv, Lk, D] bf16
 *   v   [B, Hkv, Lk, D] bf16
 *   o   [B, Hq,  Lq, D] fp32   (output)
 *   lse [B, Hq,  Lq]    fp32   (output, natural log)
 *
 * softmax_scale multiplies Q K^T (1/sqrt(D) is the usual choice, sec. 2
 * "Why divide by sqrt d?").  Uses no memory beyond its arguments.
 */
fa_status_t fa_fwd(const void* q, const void* k, const void* v, float* o, float* lse,
                   int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal,
                   float softmax_scale, cudaStream_t stream);

/*
 * Variable-length (packed) attention forward: num_seqs independent problems
 * stored back to back, token-major.
 *
 *   q   [total_q, Hq,  D] bf16;  k, v [total_k, Hkv, D] bf16
 *   o   [total_q, Hq,  D] fp32   (output)
 *   lse [Hq, total_q]     fp32   (output, natural log)
 *   cu_seqlens_q, cu_seqlens_k: int32 DEVICE arrays of num_seqs + 1
 *     non-decreasing prefix offsets starting at 0, ending at total_q / total_k.
 *     Sequence s owns query tokens [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key
 *     tokens [cu_seqlens_k[s], cu_seqlens_k[s+1]); the causal mask is relative
 *     to each sequence (bottom-right alignment per sequence).
 *   max_seqlen_q, max_seqlen_k: upper bounds on any sequence's length.
 *
 * Offsets are read on the device.  Offsets that are not non-decreasing, or a
 * sequence longer than its max_seqlen bound, latch FA_ERR_INVALID_ARG on the
 * device (reported by fa_check); such sequences produce no output.
 *
 * Scheduling (FlashAttention-4: Blackwell Attention Kernel Co-Design, "LPT
 * scheduling for imbalanced grids": variable-length batches are ordered by
 * work, longest first; FlashAttention from Scratch, sec. 11.5 on the tail of a
 * persistent grid): every CTA of the launch reads the offsets, sorts the
 * sequences by key length, longest first, and builds the tile list in its
 * own shared memory.  The call allocates no memory and needs no workspace.
 * A launch schedules at most FA_VARLEN_SEQS_PER_LAUNCH sequences (64 for
 * the (192, 128) head dimensions of fa_fwd_varlen_hdim); a larger batch is
 * processed by consecutive launches of that many sequences each, on
 * `stream`, each ordered longest first within itself.
 */
#define FA_VARLEN_SEQS_PER_LAUNCH 1536
fa_status_t fa_fwd_varlen(const void* q, const void* k, const void* v, float* o, float* lse,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                          int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                          int Hq, int Hkv, int D, int causal, float softmax_scale,
                          cudaStream_t stream);

/*
 * Variant of fa_fwd_varlen whose schedule lives in a fixed device array
 * (no counterpart on the pages: it changes where the schedule lives, not what
 * is computed).
 *
 * It is meant for callers that cannot call cudaMalloc on the hot path:
 * processes that hand all device memory to their own allocator up front,
 * runtimes that must not allocate while serving, or code that must not touch
 * a memory pool.  fa_fwd_varlen allocates nothing either, but builds its
 * schedule per CTA in shared memory and so splits batches of more than
 * FA_VARLEN_SEQS_PER_LAUNCH sequences into several launches.  This entry
 * point sorts the whole batch (up to FA_NOALLOC_MAX_SEQS sequences) once,
 * with a schedule kernel, into an array compiled into the library (about
 * 192 KiB, resident on every device that loads the library until the process
 * exits), and runs one attention launch over it.  Same arguments and results
 * as fa_fwd_varlen for D = 64 or 128; it calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 *  - num_seqs may be at most FA_NOALLOC_MAX_SEQS; larger batches return
 *    FA_ERR_INVALID_ARG before any device work.
 *  - The first call on a device resolves the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - All calls on a device share the one array: calls whose kernels can
 *    overlap on the GPU (different streams without ordering between them)
 *    race on it.  Order them on one stream, or use fa_fwd_varlen.
 */
#define FA_NOALLOC_MAX_SEQS 16384
fa_status_t fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, float* o, float* lse,
                                  const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                  int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                  int Hq, int Hkv, int D, int causal, float softmax_scale,
                                  cudaStream_t stream);

/*
 * Programmable variants of the forward (FlashAttention from Scratch, sec. 12
 * "Programmable attention: FlexAttention meets FA4"): which query-key pairs
 * may attend, and a modification of the score before the softmax.
 *
 *   window_left, window_right: key j may attend query i iff
 *       c_i - window_left <= j <= c_i + window_right,  c_i = i + (Lk - Lq)
 *     (c_i is the query's position in the key sequence, bottom-right
 *     aligned as for the causal mask; per sequence for packed batches).
 *     A negative bound is unlimited: (-1, -1) is full attention, (-1, 0) the
 *     causal mask, (w - 1, 0) a causal sliding window of width w.  KV tiles
 *     outside every row's window are skipped.
 *   softcap > 0: the scaled score s becomes softcap * tanh(s / softcap).
 *   alibi_slopes: DEVICE fp32 [Hq] (or NULL); the score of query head h
 *     becomes s - alibi_slopes[h] * |c_i - j|.
 *   Order: scale, then soft-capping, then the ALiBi bias, then the window:
 *   with both modifiers the score is softcap * tanh(s / softcap) -
 *   alibi_slopes[h] * |c_i - j| (the bias stays unbounded by the cap).
 *   D must be 64 or 128.  LSE is the log-sum-exp of the modified scores.
 */
typedef struct fa_variant {
    int window_left;
    int window_right;
    float softcap;
    const float* alibi_slopes;
} fa_variant_t;

/*
 * Forward with a value head dimension that differs from the query/key one
 * (FlashAttention-4: Blackwell Attention Kernel Co-Design, "How we know": the
 * (192, 128) case of its benchmarks, as in DeepSeek-V3-style attention).
 *
 *   q [B, Hq, Lq, D], k [B, Hkv, Lk, D], v [B, Hkv, Lk, Dv] bf16 (DEVICE)
 *   o [B, Hq, Lq, Dv] fp32, lse [B, Hq, Lq] fp32 (DEVICE, outputs)
 *
 * O = softmax(scale * Q K^T + M) V; everything else (causal rule, GQA,
 * empty rows, errors, ownership) as fa_fwd.  Supported (D, Dv): (64, 64),
 * (128, 128) and (192, 128); other pairs return FA_ERR_UNSUPPORTED.
 * fa_fwd(..., D, ...) is fa_fwd_hdim(..., D, D, ...).  1 kernel.
 */
fa_status_t fa_fwd_hdim(const void* q, const void* k, const void* v, float* o, float* lse,
                        int B, int Hq, int Hkv, int Lq, int Lk, int D, int Dv, int causal,
                        float softmax_scale, cudaStream_t stream);

/* fa_fwd_varlen with value head dimension Dv: q, k [total, H, D], v [total_k, Hkv, Dv],
 * o [total_q, Hq, Dv]; same (D, Dv) pairs as fa_fwd_hdim.  2 kernels. */
fa_status_t fa_fwd_varlen_hdim(const void* q, const void* k, const void* v, float* o, float* lse,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                               int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                               int Hq, int Hkv, int D, int Dv, int causal, float softmax_scale,
                               cudaStream_t stream);

/* fa_fwd with a variant (same layouts; `variant` is a HOST pointer). */
fa_status_t fa_fwd_variant(const void* q, const void* k, const void* v, float* o, float* lse,
                           int B, int Hq, int Hkv, int Lq, int Lk, int D, const fa_variant_t* variant,
                           float softmax_scale, cudaStream_t stream);

/* fa_fwd_varlen with a variant (windows and ALiBi distances per sequence). */
fa_status_t fa_fwd_varlen_variant(const void* q, const void* k, const void* v, float* o, float* lse,
                                  const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                  int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                  int Hq, int Hkv, int D, const fa_variant_t* variant,
                                  float softmax_scale, cudaStream_t stream);

/*
 * FP8 forward (FlashAttention from Scratch, sec. 10.3 "Treat FP8 as a second
 * lesson"; FlashAttention 1-4, FA3 item 3 "FP8 with block quantization and
 * incoherent processing").  Two steps:
 *
 * fa_fp8_prepare: rotates Q and K by the same orthogonal matrix
 *   M = diag(signs) H / sqrt(128) (H the Sylvester Hadamard matrix, applied as
 *   a fast Walsh-Hadamard transform; (QM)(KM)^T = QK^T), then quantises each
 *   128-row tile of every (batch, head) slice of QM and KM to e4m3 with scale
 *   amax(tile) / 448.  V gets one scale per (batch, KV head) slice and is
 *   stored transposed.  q, k, v: bf16 DEVICE, layouts as fa_fwd; signs: DEVICE
 *   fp32 [128], each +1 or -1 (the caller draws them).  `prepared`: caller-owned
 *   DEVICE buffer of fa_fp8_workspace bytes, 16-byte aligned.  3 kernels and a
 *   memset on `stream`.
 *
 * fa_fwd_fp8: attention of the prepared inputs: S = (QM)(KM)^T from e4m3
 *   operands on the tensor cores (kind::f8f6f4), fp32 online softmax, P
 *   rounded to e4m3 for P.V, O = (P.V) * scale_v / sum(P) in fp32.  Same
 *   output layouts, causal rule and empty-row convention as fa_fwd.  1 kernel.
 *
 * D must be 128 (FA_ERR_UNSUPPORTED otherwise).  The prepared buffer holds,
 * each section 256-byte aligned: Q codes [B*Hq][Lq][128], K codes
 * [B*Hkv][Lk][128], V codes [B*Hkv][128][Lk rounded up to 128], Q tile scales
 * [B*Hq][ceil(Lq/128)], K tile scales [B*Hkv][ceil(Lk/128)], V scales
 * [B*Hkv] (fp32), and 4 bytes per V slice of scratch.
 */
fa_status_t fa_fp8_workspace(int B, int Hq, int Hkv, int Lq, int Lk, int D, size_t* bytes);
fa_status_t fa_fp8_prepare(const void* q, const void* k, const void* v, const float* signs,
                           int B, int Hq, int Hkv, int Lq, int Lk, int D, void* prepared,
                           size_t prepared_bytes, cudaStream_t stream);
fa_status_t fa_fwd_fp8(const void* prepared, float* o, float* lse, int B, int Hq, int Hkv,
                       int Lq, int Lk, int D, int causal, float softmax_scale, cudaStream_t stream);

/*
 * Split-KV forward for decode (FlashAttention from Scratch, sec. 9.1 "Split
 * the long dimension that remains"; sec. 4.3 "Merge independently computed
 * partitions").  Same operation, layouts and causal rule as fa_fwd, for
 * problems with few query rows per KV head and a long key range: the key
 * range of every (batch, KV head) is cut into num_splits partitions that run
 * as independent CTAs, each producing a normalised partial output and its
 * log-sum-exp, and a second kernel merges the partitions by their softmax
 * mass.  All (Hq / Hkv) * Lq query rows that share a KV head are served by
 * one pass over its K and V.
 *
 *   q   [B, Hq,  Lq, D] bf16;  k, v [B, Hkv, Lk, D] bf16
 *   o   [B, Hq,  Lq, D] fp32 (output);  lse [B, Hq, Lq] fp32 (output, natural log)
 *   (Hq / Hkv) * Lq must be at most 16, else FA_ERR_UNSUPPORTED (use fa_fwd).
 *   num_splits: partitions of the key range; <= 0 picks a count from the
 *     shape and the device's SM count; values above ceil(Lk / 64) are reduced
 *     to it (a partition holds whole 64-key tiles).
 *   workspace: caller-owned DEVICE memory of at least the size that
 *     fa_fwd_splitkv_workspace reports for the same shape and num_splits
 *     (16-byte aligned; may be NULL when that size is 0, i.e. one partition).
 *     It holds the partial results between the two kernels; no memory is
 *     allocated by the call.  Calls that overlap on the GPU need separate
 *     workspaces.
 *
 * Launches 1 kernel (one partition) or 2 (partials, then the merge).
 * Scores, softmax statistics and O accumulate in fp32; the tensor-core
 * partials ((Hq / Hkv) * Lq >= 2, D = 64 or 128) round P to bf16 for P.V, as
 * fa_fwd does, and the one-row kernel keeps P in fp32.
 */
fa_status_t fa_fwd_splitkv(const void* q, const void* k, const void* v, float* o, float* lse,
                           int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal,
                           float softmax_scale, int num_splits, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes fa_fwd_splitkv needs for this shape and num_splits on the
 * CURRENT device (the automatic count depends on its SM count), written to
 * *workspace_bytes; *splits_used (if not NULL) receives the partition count
 * the call will use.  Same argument checks as fa_fwd_splitkv.
 */
fa_status_t fa_fwd_splitkv_workspace(int B, int Hq, int Hkv, int Lq, int Lk, int D, int num_splits,
                                     size_t* workspace_bytes, int* splits_used);

/*
 * Attention backward (FlashAttention from Scratch, sec. 8 "Backward: spend
 * arithmetic to save memory").  Given the forward's inputs, its output O and
 * log-sum-exp LSE (as written by fa_fwd) and the upstream gradient dO, returns
 * the gradients of sum(O * dO):
 *
 *     dV = P^T dO,  dS = P * (dO V^T - rowsum(O * dO)),  dQ = c dS K,  dK = c dS^T Q
 *
 * with P rebuilt from Q, K and LSE (never stored) and c = softmax_scale.
 * Grouped-query heads add into their shared KV head.  Same masking rules as
 * fa_fwd; rows with LSE = -inf contribute nothing.
 *
 *   q [B, Hq, Lq, D], k/v [B, Hkv, Lk, D], dout [B, Hq, Lq, D]: bf16
 *   o [B, Hq, Lq, D], lse [B, Hq, Lq]: fp32 (fa_fwd's outputs)
 *   dq [B, Hq, Lq, D], dk/dv [B, Hkv, Lk, D]: fp32 outputs, fully overwritten
 *   workspace: DEVICE memory of at least fa_bwd_workspace bytes, 16-byte
 *     aligned, owned by the caller (per-row statistics between the two
 *     kernels); calls that overlap on the GPU need separate workspaces.
 *   D must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 *
 * Launches 2 kernels: a preprocess (rowsum(O * dO), LSE in base 2, dq zeroed)
 * and the gradient kernel.  dq is accumulated by fp32 reduce-adds (the TMA's
 * atomic additions) from several CTAs in no fixed order, so its low bits may
 * differ between runs; dk and dv are deterministic.
 */
fa_status_t fa_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse,
                   const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Lq,
                   int Lk, int D, int causal, float softmax_scale, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes fa_bwd needs: 8 * B * Hq * (Lq rounded up to 128), written to *workspace_bytes. */
fa_status_t fa_bwd_workspace(int B, int Hq, int Lq, size_t* workspace_bytes);

/*
 * Backward of a packed (variable-length) batch: the gradients of fa_fwd_varlen,
 * each sequence an independent problem with its own bottom-right causal
 * alignment.
 *
 *   q, dout [total_q, Hq, D], k, v [total_k, Hkv, D]: bf16
 *   o [total_q, Hq, D], lse [Hq, total_q]: fp32 (fa_fwd_varlen's outputs)
 *   dq [total_q, Hq, D], dk/dv [total_k, Hkv, D]: fp32 outputs, fully
 *     overwritten (zero for sequences without keys / without query rows)
 *   cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k: as fa_fwd_varlen
 *     (invalid offsets latch FA_ERR_INVALID_ARG on the device, read by fa_check)
 *   workspace: DEVICE memory of at least fa_bwd_varlen_workspace bytes,
 *     16-byte aligned, owned by the caller (row statistics and the schedule);
 *     calls that overlap on the GPU need separate workspaces.
 *   D must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 *
 * Launches 3 kernels: the schedule (sequences longest query range first), the
 * preprocess and the gradient kernel.  No device memory is allocated.
 */
fa_status_t fa_bwd_varlen(const void* q, const void* k, const void* v, const float* o, const float* lse,
                          const void* dout, float* dq, float* dk, float* dv, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, int num_seqs, int total_q, int total_k,
                          int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D, int causal,
                          float softmax_scale, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* Workspace bytes fa_bwd_varlen needs for num_seqs sequences of total_q query
 * tokens and Hq query heads, written to *workspace_bytes. */
fa_status_t fa_bwd_varlen_workspace(int num_seqs, int total_q, int Hq, size_t* workspace_bytes);

/*
 * Backward of fa_fwd_variant / fa_fwd_varlen_variant for key windows,
 * soft-capping and ALiBi (FlashAttention from Scratch, sec. 12): the same
 * modified scores t and masks as the forward (pass the forward's O and LSE).
 * The gradient with respect to t is P * (dP - delta); the ALiBi bias and the
 * masks do not depend on the raw score s, so that is dS, while soft-capping
 * (t = cap * tanh(s / cap)) multiplies it by dt/ds = 1 - tanh^2(s / cap).
 * With both modifiers the factor dt/ds is that of the cap alone.  Layouts,
 * workspace and launches as fa_bwd / fa_bwd_varlen; `variant` is a HOST
 * pointer.  D must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 */
fa_status_t fa_bwd_variant(const void* q, const void* k, const void* v, const float* o, const float* lse,
                           const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Lq,
                           int Lk, int D, const fa_variant_t* variant, float softmax_scale, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);
fa_status_t fa_bwd_varlen_variant(const void* q, const void* k, const void* v, const float* o, const float* lse,
                                  const void* dout, float* dq, float* dk, float* dv, const int* cu_seqlens_q,
                                  const int* cu_seqlens_k, int num_seqs, int total_q, int total_k,
                                  int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                  const fa_variant_t* variant, float softmax_scale, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device-side error latch
 * of the current device: FA_ERR_TIMEOUT or FA_ERR_INVALID_ARG from an earlier
 * launch, or FA_ERR_CUDA when a kernel found its launch configuration unusable
 * and did nothing; FA_ERR_CUDA also if the stream reports an error.
 */
fa_status_t fa_check(cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status_t status);

/*
 * Number of kernels the last successful forward call on this host thread
 * launched (1 for dense, 2 for varlen: schedule + attention; 1 or 2 for
 * split-KV: partials, then the merge when there is more than one partition;
 * 2 for backward).
 */
int fa_last_launch_count(void);

/*
 * Test hook (no counterpart on the pages).  kind = 1 makes the next fa_fwd
 * (or fa_fwd_splitkv, fa_bwd or fa_fwd_fp8) call on this host thread drop the first K
 * tile load (split-KV, backward: the first K/V tile) of every CTA: the bounded wait for it runs out (about 1 s), every thread of
 * the kernel retires, and fa_check then reports FA_ERR_TIMEOUT with the CUDA
 * context still usable.  kind = 0 clears a pending request.  Results of the faulted
 * call are undefined.
 */
void fa_test_inject_fault(int kind);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
