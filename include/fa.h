/*
 * fa.h -- C ABI of libfa.so: numerically stable row softmax and exact fused
 * attention forward (online softmax, FlashAttention-style) for one NVIDIA
 * GB300 (sm_103a).
 *
 * The operations are defined on these pages:
 *   [L22] "第二十二课：Softmax 为什么难以高效，以及 FlashAttention 如何减少显存访问"
 *         (lincklin.cn, lesson 22)
 *   [FG]  "少搬一趟：FlashAttention 四代进化史" (chengshu-blog booklet)
 *   [OF]  "从 FlashAttention 看懂算子融合：为什么融合、少读写了什么、又会错在哪里"
 *         (jokeuncle.github.io notes)
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller (for
 *     example memory allocated through PyTorch).  The library never frees or
 *     keeps them; it allocates no device memory per call.
 *   - Work is enqueued on the library stream of the calling thread (see
 *     fa_set_stream) and the call returns without synchronising, except where
 *     a function says otherwise.  A return value of FA_OK means the work was
 *     launched; faults inside a kernel surface at the caller's next
 *     synchronisation, and timeouts of the kernels' internal waits are
 *     reported by fa_get_device_error.
 *   - A negative return value means nothing was launched.
 *   - The library is thread-compatible: the stream setting is per host thread.
 *   - Per-device state (the device error word's address, the static scratch
 *     array's address, the helper streams of fa_attention_fwd_host) is looked
 *     up once per device and kept for the life of the process.  A device reset
 *     (cudaDeviceReset) or the destruction of the primary context invalidates
 *     it: after either, make no further call into the library in that process.
 */
#ifndef FA_H_
#define FA_H_

#include <stdint.h>

/* Entry points keep default visibility; everything else in the library is hidden. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes --------------------------------------------------------- */
#define FA_OK 0
#define FA_ERR_NULL_POINTER (-1)    /* a required pointer is NULL               */
#define FA_ERR_BAD_SIZE (-2)        /* a size is negative or inconsistent         */
#define FA_ERR_UNSUPPORTED (-3)     /* head dimension or option not supported     */
#define FA_ERR_MISALIGNED (-4)      /* a pointer breaks the alignment rule        */
#define FA_ERR_CUDA (-5)            /* a CUDA runtime/driver call failed          */
#define FA_ERR_TOO_LARGE (-6)       /* a size exceeds what the kernels index      */
#define FA_ERR_NO_DEVICE (-7)       /* no usable sm_103 device is current         */
#define FA_ERR_SCRATCH_LIMIT (-8)   /* needs more than the library's static scratch */

/* ---- device error word bits (fa_get_device_error) ------------------------- */
#define FA_DEVERR_WAIT_TIMEOUT 0x1  /* a pipeline wait gave up (bounded wait)     */
#define FA_DEVERR_BAD_SEQLENS 0x2   /* cu_seqlens disagreed with N or the tensors */

/*
 * Row softmax, numerically stable ([L22] §二 "数值稳定 Softmax": shift by the
 * row maximum; §三 the max / exp-sum / normalise steps; §六–§十 warp-per-row
 * and block-per-row reductions):
 *     y[r, j] = exp(x[r, j] - m_r) / sum_k exp(x[r, k] - m_r),  m_r = max_k x[r, k]
 *
 *   x     fp32 [rows, N], row-major, contiguous (row stride N elements).
 *   y     fp32 [rows, N], same layout.  y == x (in place) is allowed; any other
 *         overlap is not.
 *   rows  number of rows, >= 0 (0 launches nothing and returns FA_OK).
 *   N     row length, >= 0 (0 launches nothing).  rows * N < 2^62.
 * Pointers need 4-byte alignment; 16-byte aligned pointers with N % 4 == 0 take
 * the vectorised path.  A row with a NaN yields NaN; a row of only -inf yields
 * NaN (0/0 in the definition).
 * Errors: FA_ERR_NULL_POINTER (x or y NULL with rows*N > 0), FA_ERR_BAD_SIZE
 * (negative size), FA_ERR_MISALIGNED, FA_ERR_CUDA.
 */
FA_API int fa_softmax_rows(const float *x, float *y, int64_t rows, int64_t N);

/*
 * Exact attention forward, bf16 in / bf16 out, fp32 accumulation, on the
 * tensor cores (tcgen05 + TMEM, TMA-fed):
 *     S = scale * Q K^T (+ mask),  P = softmax(S) row-wise,  O = P V,
 *     lse[i] = log(sum_j exp(S[i, j]))  (natural log)
 * computed tile by tile with the online-softmax recurrence ([L22] §三十二
 * pseudo-code; [FG] §2.2 update of m, l and the unnormalised output, §3.2
 * deferred normalisation, §2.4 logsumexp; [OF] "FlashAttention 的核心变化")
 * without materialising S or P in device memory.
 *
 * Layouts (all contiguous, row-major):
 *   dense  (cu_seqlens == NULL): Q, K, V, O  [B, N, H, d];  lse [B, H, N].
 *   packed (cu_seqlens != NULL): Q, K, V, O  [total, H, d]; lse [H, total];
 *          sequence b owns tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 ([L22] §三十五
 *          "Packed Sequence / Variable-Length"); B = number of sequences,
 *          N = longest sequence length (an upper bound is fine).
 *   Q, K, V, O: bf16 (raw 16-bit storage); lse: fp32.
 *   cu_seqlens: DEVICE int32 [B + 1], non-decreasing, cu_seqlens[0] = 0.
 *   d: 64 or 128.  scale: multiplies Q K^T (1/sqrt(d) for standard attention).
 *   causal != 0: query i sees keys j <= i of its own sequence ([L22] §三十四).
 * Alignment: Q, K, V, O 16-byte aligned; lse 4-byte aligned.
 * The packed form reads total = cu_seqlens[B] back to the host and therefore
 * synchronises the library stream once per call (fa_attention_fwd_varlen takes
 * total from the caller and does not).  A sequence longer than N is not
 * computed and sets FA_DEVERR_BAD_SEQLENS in the device error word.
 * Errors: FA_ERR_NULL_POINTER, FA_ERR_BAD_SIZE, FA_ERR_UNSUPPORTED (d),
 * FA_ERR_MISALIGNED, FA_ERR_TOO_LARGE, FA_ERR_NO_DEVICE, FA_ERR_CUDA.
 */
FA_API int fa_attention_fwd(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                     int H, int N, int d, float scale, int causal, const int32_t *cu_seqlens);

/*
 * Same as fa_attention_fwd with packed sequences, with the packed token count
 * `total` (= cu_seqlens[B]) given by the caller: nothing is read back and the
 * call does not synchronise.  cu_seqlens must not be NULL.
 */
FA_API int fa_attention_fwd_varlen(const void *Q, const void *K, const void *V, void *O, float *lse,
                            int B, int H, int N, int64_t total, int d, float scale, int causal,
                            const int32_t *cu_seqlens);

/*
 * Split-KV attention forward ("从 FlashAttention 看懂算子融合…": split the keys of a
 * query block, keep per-split outputs and logsumexps, merge them in a combine
 * kernel; the merge is the online-softmax rule of [L22] §十九 / §二十二).  For
 * problems whose (sequence, head, 256-query block) count is too small to fill
 * the GPU, e.g. a short block of new queries against a long context.
 *
 *   Q, O: bf16 [B, Nq, H, d];  K, V: bf16 [B, Nk, H, d];  lse: fp32 [B, H, Nq].
 *   causal != 0: the queries are the last Nq positions of each sequence of Nk
 *   keys (bottom-right alignment): query i sees keys j <= i + Nk - Nq; needs
 *   Nk >= Nq.  With Nq == Nk this is fa_attention_fwd's masking.
 *   num_splits: key ranges per query block; 0 lets the library choose
 *   (fa_splitkv_num_splits); values above ceil(Nk / 128) are clamped.
 *   O_accum: fp32 [num_splits, B, Nq, H, d] and lse_accum: fp32
 *   [num_splits, B, H, Nq] -- DEVICE scratch owned by the caller, 16-byte and
 *   4-byte aligned; contents on entry are ignored.  Unused (may be NULL) when
 *   the split count in effect is 1.  Sizes use the split count in effect.
 *   d: 64 or 128; Q, K, V, O 16-byte aligned.
 * Runs the tensor-core kernel on every (block, split) and, when splits > 1,
 * the combine kernel; no synchronisation.
 * Errors: as fa_attention_fwd, and FA_ERR_BAD_SIZE for causal with Nk < Nq or
 * num_splits < 0, FA_ERR_NULL_POINTER for missing scratch.
 */
FA_API int fa_attention_fwd_splitkv(const void *Q, const void *K, const void *V, void *O,
                                    float *lse, int B, int H, int Nq, int Nk, int d, float scale,
                                    int causal, int num_splits, float *O_accum, float *lse_accum);

/*
 * fa_attention_fwd_splitkv for packed sequences whose query and key counts
 * differ per sequence ("第二十二课…" §三十五 packed / variable-length sequences;
 * e.g. one decode step over caches of different lengths): sequence b owns
 * query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows
 * cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 and attends to nothing else.
 *   Q, O: bf16 [total_q, H, d];  K, V: bf16 [total_k, H, d];  lse: fp32
 *   [H, total_q].  cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B + 1], each
 *   non-decreasing from 0 to total_q / total_k.  Nq, Nk: the longest query
 *   and key counts (upper bounds are fine; they size the grid and the split
 *   choice).  causal != 0: within each sequence bottom-right aligned, query i
 *   sees keys j <= i + Lk - Lq; a sequence with Lk < Lq, or longer than Nq /
 *   Nk, is not computed and sets FA_DEVERR_BAD_SEQLENS.
 *   num_splits: as fa_attention_fwd_splitkv (0: the library chooses from B,
 *   H, Nq, Nk).  O_accum: fp32 [num_splits, total_q, H, d], lse_accum: fp32
 *   [num_splits, H, total_q] -- caller scratch as in fa_attention_fwd_splitkv
 *   (unused when one split is in effect).  Nothing is read back; no
 *   synchronisation.
 * Errors: as fa_attention_fwd_splitkv, and FA_ERR_NULL_POINTER for a NULL
 * prefix-sum array.
 */
FA_API int fa_attention_fwd_splitkv_varlen(const void *Q, const void *K, const void *V, void *O,
                                           float *lse, int B, int H, int Nq, int Nk,
                                           int64_t total_q, int64_t total_k, int d, float scale,
                                           int causal, int num_splits,
                                           const int32_t *cu_seqlens_q,
                                           const int32_t *cu_seqlens_k, float *O_accum,
                                           float *lse_accum);

/*
 * Attention backward for the bf16 forward (dense batches): the gradients of
 * sum(dO * O) with respect to Q, K and V, with the probabilities recomputed
 * from the forward's row logsumexp ("少搬一趟…" §2.4: P_ij = exp(S_ij - L_i);
 * "第二十二课…" §三十-三十一) and the chain rule written out:
 *     dV = P^T dO,  dS = P o (dO V^T - D),  D_i = dO_i . O_i,
 *     dQ = scale dS K,  dK = scale dS^T Q.
 *   Q, K, V, O, dO: bf16 [B, N, H, d] (O and lse as written by fa_attention_fwd
 *   for the same Q, K, V, scale and causal); lse: fp32 [B, H, N].
 *   dQ, dK, dV: bf16 [B, N, H, d], written.
 *   D_buf: fp32 [B, H, N] DEVICE scratch owned by the caller (receives D_i;
 *   contents on entry are ignored).
 *   d: 64 or 128; bf16 pointers 16-byte aligned, lse and D_buf 4-byte aligned.
 * Two kernels run on the library stream (dQ and D, then dK and dV); no
 * synchronisation.  Packed batches: fa_attention_bwd_varlen.
 * Errors: FA_ERR_NULL_POINTER, FA_ERR_BAD_SIZE, FA_ERR_UNSUPPORTED (d),
 * FA_ERR_MISALIGNED, FA_ERR_TOO_LARGE, FA_ERR_NO_DEVICE, FA_ERR_CUDA.
 */
FA_API int fa_attention_bwd(const void *Q, const void *K, const void *V, const void *O,
                            const void *dO, const float *lse, void *dQ, void *dK, void *dV,
                            float *D_buf, int B, int H, int N, int d, float scale, int causal);

/*
 * fa_attention_bwd for packed sequences ("第二十二课…" §三十五: a batch of
 * variable-length sequences stored one after another, none attending to
 * another): each sequence's gradients are those of its own attention.
 *   Q, K, V, O, dO, dQ, dK, dV: bf16 [total, H, d]; lse and D_buf: fp32
 *   [H, total] (the layout fa_attention_fwd writes lse in for packed
 *   batches); cu_seqlens: DEVICE int32 [B + 1], non-decreasing, from 0 to
 *   total; N: the longest sequence (an upper bound is fine); total: the
 *   packed row count (= cu_seqlens[B]; nothing is read back, no
 *   synchronisation).  A sequence longer than N is not computed and sets
 *   FA_DEVERR_BAD_SEQLENS in the device error word.
 * Errors: as fa_attention_bwd, and FA_ERR_NULL_POINTER for a NULL cu_seqlens.
 */
FA_API int fa_attention_bwd_varlen(const void *Q, const void *K, const void *V, const void *O,
                                   const void *dO, const float *lse, void *dQ, void *dK,
                                   void *dV, float *D_buf, int B, int H, int N, int64_t total,
                                   int d, float scale, int causal, const int32_t *cu_seqlens);

/*
 * fa_attention_bwd in one pass over the key tiles, with dQ summed by atomic
 * adds ("少搬一趟…" §3.3: the backward is split along the K, V column blocks,
 * one block per CTA, and the blocks' overlapping contributions to dQ are
 * summed with atomic additions; §5.6).  Each CTA forms dK and dV of its 128
 * keys and its share dS K of dQ for every 64 queries it sees; the shares are
 * added in fp32 into `workspace` by atomic adds (performed in L2), and a last
 * kernel writes dQ = scale * sum in bf16.  S and dP are formed once (five
 * products instead of fa_attention_bwd's seven).
 *   Arguments, layouts and the result's definition: as fa_attention_bwd
 *   (dense batches; D_buf receives D_i).  d: 64 or 128.
 *   workspace: DEVICE scratch owned by the caller, 256-byte aligned, at least
 *   fa_attention_bwd_atomic_workspace_bytes(B, H, N, d) bytes: the fp32 dQ
 *   accumulator [B * H, n_pad, d], then fp32 (lse log2 e, D) pairs [B * H,
 *   n_pad], n_pad = N rounded up to 64; contents on entry are ignored (the
 *   first kernel writes all of it).
 * The order of the atomic adds is not fixed, so dQ may differ from run to run
 * in its last bits; dK and dV are reproducible.  fa_attention_bwd is the
 * deterministic form ("少搬一趟…" §5.6 offers one for the same reason).
 * Three kernels run on the library stream (D_i and zeroing, the pass, the dQ
 * conversion); no synchronisation.
 * Errors: as fa_attention_bwd; FA_ERR_BAD_SIZE also for a workspace that is
 * too small.
 */
FA_API int fa_attention_bwd_atomic(const void *Q, const void *K, const void *V, const void *O,
                                   const void *dO, const float *lse, void *dQ, void *dK,
                                   void *dV, float *D_buf, int B, int H, int N, int d,
                                   float scale, int causal, void *workspace,
                                   int64_t workspace_bytes);

/* Workspace bytes fa_attention_bwd_atomic needs, or a negative FA_ERR_* code. */
FA_API int64_t fa_attention_bwd_atomic_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_attention_bwd_atomic for packed sequences ("第二十二课…" §三十五 with
 * "少搬一趟…" §3.3): each sequence's gradients are those of its own attention.
 *   Q, K, V, O, dO, dQ, dK, dV: bf16 [total, H, d]; lse and D_buf: fp32
 *   [H, total]; cu_seqlens: DEVICE int32 [B + 1], non-decreasing from 0 to
 *   total; N: the longest sequence (an upper bound is fine); d: 64 or 128.
 *   workspace: DEVICE scratch owned by the caller, 256-byte aligned, at least
 *   fa_attention_bwd_atomic_varlen_workspace_bytes(B, H, N, total, d) bytes:
 *   the fp32 dQ accumulator [H, total + 64, d], then fp32 (lse log2 e, D)
 *   pairs [H, B, n_pad] (n_pad = N rounded up to 64); contents on entry are
 *   ignored.  A sequence longer than N is not computed and sets
 *   FA_DEVERR_BAD_SEQLENS.  dQ's last bits may differ from run to run.
 * Errors: as fa_attention_bwd_atomic, and FA_ERR_NULL_POINTER for a NULL
 * cu_seqlens.
 */
FA_API int fa_attention_bwd_atomic_varlen(const void *Q, const void *K, const void *V,
                                          const void *O, const void *dO, const float *lse,
                                          void *dQ, void *dK, void *dV, float *D_buf, int B,
                                          int H, int N, int64_t total, int d, float scale,
                                          int causal, const int32_t *cu_seqlens, void *workspace,
                                          int64_t workspace_bytes);

/* Workspace bytes fa_attention_bwd_atomic_varlen needs, or a negative FA_ERR_* code. */
FA_API int64_t fa_attention_bwd_atomic_varlen_workspace_bytes(int B, int H, int N, int64_t total,
                                                              int d);

/*
 * FP8 attention forward ("少搬一趟…" §4.6: FP8 with blockwise quantisation and
 * incoherent processing), for bf16 inputs on dense batches:
 *   1. Q and K rows are multiplied by M = diag(signs) H_d / sqrt(d) (H_d the
 *      Sylvester-Hadamard matrix): (QM)(KM)^T = Q K^T, large components spread
 *      over the row;
 *   2. each 128-row tile of a head of QM and KM, and each head of V, gets a
 *      scale amax / 448 and is rounded to e4m3 (nearest even, saturating);
 *   3. the attention runs on the tensor cores with e4m3 operands (P also in
 *      e4m3), fp32 accumulation, the scales folded back in; O is bf16.
 *   Q, K, V, O: bf16 [B, N, H, d]; lse: fp32 [B, H, N] (natural log);
 *   causal: key j visible to query i iff j <= i.
 *   signs: DEVICE fp32 [d] of +1 / -1 (the random signs of M, drawn by the
 *   caller; any fixed draw gives the same result up to rounding).
 *   workspace: DEVICE scratch owned by the caller, 256-byte aligned, at least
 *   fa_attention_fp8_workspace_bytes(B, H, N, d) bytes; contents on entry are
 *   ignored.  It receives, in this order, each part starting on a 256-byte
 *   boundary (T = ceil(N / 128)): e4m3 Q M / sq [B*N, H, d], e4m3 K M / sk
 *   [B*N, H, d], e4m3 V^T / sv [B, H, d, 128 T], fp32 sq and sk [B, H, T],
 *   fp32 per-tile amax of V [B, H, T], fp32 sv [B, H].
 *   d: 128 only.  Size limits: ceil(N / 128) <= 65535 and
 *   3 * B * H * ceil(N / 128) < 2^31 (FA_ERR_TOO_LARGE otherwise).
 *   Packed batches: fa_attention_fwd_fp8_varlen.
 * Three kernels run on the library stream; no synchronisation.
 * Errors: FA_ERR_UNSUPPORTED (d != 128), FA_ERR_BAD_SIZE (also a workspace
 * that is too small), FA_ERR_NULL_POINTER, FA_ERR_MISALIGNED, FA_ERR_TOO_LARGE,
 * FA_ERR_NO_DEVICE, FA_ERR_CUDA.
 */
FA_API int fa_attention_fwd_fp8(const void *Q, const void *K, const void *V, void *O, float *lse,
                                int B, int H, int N, int d, float scale, int causal,
                                const float *signs, void *workspace, int64_t workspace_bytes);

/* Workspace bytes fa_attention_fwd_fp8 needs, or a negative FA_ERR_* code. */
FA_API int64_t fa_attention_fp8_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_attention_fwd_fp8 for packed sequences ("第二十二课…" §三十五: variable-length
 * sequences stored one after another, none attending to another).  Each
 * sequence is quantised on its own: Q and K tiles of 128 rows from the
 * sequence's first token (a tile cut by the sequence's end takes its amax over
 * the sequence's rows only), one V scale per (sequence, head).
 *   Q, K, V, O: bf16 [total, H, d]; lse: fp32 [H, total]; cu_seqlens: DEVICE
 *   int32 [B + 1], non-decreasing from 0 to total; N: the longest sequence (an
 *   upper bound is fine; it sizes the tile grid and the workspace); total: the
 *   packed row count (= cu_seqlens[B]; nothing is read back).
 *   workspace: at least fa_attention_fp8_varlen_workspace_bytes(B, H, N, total,
 *   d) bytes, laid out as for the dense call with [total, H, d] code arrays
 *   and per-sequence padded V'^T [B, H, d, 128 ceil(N / 128)].
 *   causal: key j of a sequence visible to its query i iff j <= i.
 * A sequence longer than N is not computed and sets FA_DEVERR_BAD_SEQLENS.
 * Errors: as fa_attention_fwd_fp8, and FA_ERR_NULL_POINTER for a NULL
 * cu_seqlens.
 */
FA_API int fa_attention_fwd_fp8_varlen(const void *Q, const void *K, const void *V, void *O,
                                       float *lse, int B, int H, int N, int64_t total, int d,
                                       float scale, int causal, const int32_t *cu_seqlens,
                                       const float *signs, void *workspace,
                                       int64_t workspace_bytes);

/* Workspace bytes fa_attention_fwd_fp8_varlen needs, or a negative FA_ERR_* code. */
FA_API int64_t fa_attention_fp8_varlen_workspace_bytes(int B, int H, int N, int64_t total, int d);

/*
 * bf16 attention forward on HOST buffers: the same result as fa_attention_fwd
 * on a dense batch (bit for bit: the same kernel runs on each head), with the
 * host <-> device copies inside the call and overlapped with the work.  The
 * pages' method is unchanged; they say nothing of where the tensors live, so
 * this entry point is the library's own (offload of whole batches).
 *   Q, K, V: HOST bf16 [B, N, H, d], read; O: HOST bf16 [B, N, H, d] and lse:
 *   HOST fp32 [B, H, N], written.  Page-locked (pinned) host memory is needed
 *   for the copies to overlap anything; pageable memory still works.
 *   workspace: DEVICE scratch owned by the caller, 256-byte aligned, at least
 *   fa_attention_host_workspace_bytes(B, H, N, d) bytes (device copies of Q,
 *   K, V, O and lse); contents on entry are ignored.
 *   d: 64 or 128.
 * The heads are taken in groups: for each group a strided copy brings its
 * slices of Q, K and V to the device (one stream), the attention kernel runs
 * on that head range (the library stream), and its slices of O and lse go
 * back (a third stream), so the copies of one group overlap the work and the
 * copies of the others.  Every operation is ordered after the work already on
 * the library stream, and the library stream waits for the last copy: the
 * call is asynchronous like the others, and O and lse are complete once the
 * library stream has been synchronised.  Every argument is checked before
 * anything is enqueued; if a CUDA call fails after copies were enqueued, the
 * library stream is still made to wait for them before the error returns, so
 * synchronising it before freeing Q, K, V suffices on every path.  The helper
 * streams and events are created once per device; concurrent calls from
 * several threads must not overlap.
 * Errors: FA_ERR_NULL_POINTER, FA_ERR_BAD_SIZE (also a workspace that is too
 * small), FA_ERR_UNSUPPORTED (d), FA_ERR_MISALIGNED (workspace), FA_ERR_TOO_LARGE,
 * FA_ERR_NO_DEVICE, FA_ERR_CUDA.
 */
FA_API int fa_attention_fwd_host(const void *Q, const void *K, const void *V, void *O, float *lse,
                                 int B, int H, int N, int d, float scale, int causal,
                                 void *workspace, int64_t workspace_bytes);

/* Workspace bytes fa_attention_fwd_host needs, or a negative FA_ERR_* code. */
FA_API int64_t fa_attention_host_workspace_bytes(int B, int H, int N, int d);

/*
 * The split count fa_attention_fwd_splitkv uses for num_splits = 0 on the
 * current device: as many splits as fill the SMs in one wave (floor of SMs /
 * 256-query blocks, 1 when the blocks alone fill more than half of the SMs),
 * at least two 128-key tiles per split.  Returns >= 1, or a negative FA_ERR_*
 * code.
 */
FA_API int fa_splitkv_num_splits(int B, int H, int Nq, int Nk, int d);

/*
 * Size in bytes of the device scratch array that
 * fa_attention_fwd_splitkv_noalloc uses (64 MiB).
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * fa_attention_fwd_splitkv without caller scratch.  The pages have no
 * counterpart to this function: it is a library convenience, not a step of
 * the method.  Same definition, arguments (minus O_accum and lse_accum),
 * masks, split choice and results as fa_attention_fwd_splitkv.
 *
 * For callers that cannot allocate device memory or pass a workspace at the
 * call site: a plug-in whose host framework hands it only its input and output
 * buffers, code that must not call cudaMalloc (which can synchronise the device
 * and can fail under memory pressure) in a latency-bound decode loop, or a
 * process whose device memory budget is fixed after start-up.  This function
 * makes no device allocation and calls no allocating routine.
 *
 * Scratch: the per-split partials live in one library-owned device array of
 * FA_NOALLOC_SCRATCH_BYTES per device, taken when the CUDA runtime loads that
 * part of the library on the device (with lazy module loading, the CUDA
 * default, at the first call of this function there) and held until the
 * context ends.  With S splits in effect a call needs
 * S * B * Nq * H * (d + 1) * 4 bytes of it; a call that needs more returns
 * FA_ERR_SCRATCH_LIMIT and launches nothing (pass a smaller num_splits, or use
 * fa_attention_fwd_splitkv with scratch of your own).  With one split in
 * effect no scratch is used.  Nothing in the array has to start at zero:
 * every element the combine reads is written earlier in the same call.
 *
 * The array's device address is looked up once per device, with that device
 * current, on the first call that needs scratch there; make that first call
 * before any stream capture begins.
 *
 * Calls share the one array per device: two calls whose work can run at the
 * same time on one device (different streams, or different host threads with
 * different streams) race on it and may return wrong results.  Calls on one
 * stream run in order and are safe.
 *
 * Errors: as fa_attention_fwd_splitkv, in the same order (except
 * FA_ERR_NULL_POINTER for scratch), then FA_ERR_SCRATCH_LIMIT as above, and
 * FA_ERR_CUDA if the array's address cannot be looked up.
 */
FA_API int fa_attention_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O,
                                            float *lse, int B, int H, int Nq, int Nk, int d,
                                            float scale, int causal, int num_splits);

/*
 * Exact attention forward in fp32 throughout (fp32 Q, K, V, O, lse), on the
 * CUDA cores, for inputs that need fp32 accuracy.  Same definition, layouts,
 * masks and cu_seqlens convention as fa_attention_fwd (the packed form reads
 * cu_seqlens[B] back and synchronises the stream once).  d: 1 .. 128.
 * Pointers 4-byte aligned.
 */
FA_API int fa_attention_fwd_f32(const float *Q, const float *K, const float *V, float *O, float *lse,
                         int B, int H, int N, int d, float scale, int causal,
                         const int32_t *cu_seqlens);

/*
 * Sets the CUDA stream (a cudaStream_t passed as void*) that later calls from
 * this host thread launch on; NULL selects the legacy default stream.  The
 * library does not take ownership.  Returns FA_OK.
 */
FA_API int fa_set_stream(void *stream);

/*
 * Failure detection, for tests: arms a wait that cannot complete in the next
 * bf16 attention forward (fa_attention_fwd / fa_attention_fwd_varlen) or
 * one-pass backward (fa_attention_bwd_atomic / fa_attention_bwd_atomic_varlen)
 * launched from this host thread, whichever comes first.  In that launch the
 * warp that issues the tensor-core instructions first waits, bounded by `ns`
 * nanoseconds, on a barrier that nothing arrives at.  The wait runs out, sets
 * FA_DEVERR_WAIT_TIMEOUT in the device error word and raises the CTA's abort
 * flag, and every CTA winds down the way it does after any timed-out wait: the
 * other roles leave their loops, copies already issued are waited for, tensor
 * memory is freed, and O and lse (forward) or dK and dV (backward) are left
 * unwritten; the backward's dQ is converted from an accumulator that received
 * nothing, so it reads zero.  The launch returns FA_OK; the error shows in
 * fa_get_device_error.  One-shot: the setting is consumed by that launch.  The
 * kernels' own waits keep their bound (2 s), so the device stays usable and the
 * next call runs normally.  ns: 1 .. 10^9 arms, 0 disarms.
 * Errors: FA_ERR_BAD_SIZE (ns < 0 or > 10^9).
 */
FA_API int fa_debug_expire_next_wait(int64_t ns);

/* The stream currently selected for this host thread. */
FA_API void *fa_get_stream(void);

/*
 * Returns the device error word of the current device (an OR of FA_DEVERR_*
 * bits raised by kernels since the last call) and clears it.  Synchronises the
 * device.  Returns a negative FA_ERR_* code if the word cannot be read.
 */
FA_API int fa_get_device_error(void);

/* Static, human-readable text for an FA_* return code. */
FA_API const char *fa_strerror(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
