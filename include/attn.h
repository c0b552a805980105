/*
 * attn.h — C ABI of the GB300 (sm_103a) exact-attention library
 * (libattn_gb300.so).
 *
 * What it computes.  Exact scaled dot-product attention,
 *     O = softmax(scale * Q K^T) V,   LSE_i = ln sum_j exp(scale * q_i . k_j),
 * evaluated tile by tile with the online-softmax recurrence (running row max,
 * rescale factor exp(m_old - m_new), running sum, unnormalised output, one
 * final division), so the score and probability matrices never reach device
 * memory.  Definitions: "TileLang tutorial, ch.15 Operators: Attention",
 * sections 1.1 and 2.1-2.5; "llm-course, ch.19 Flash Attention", sections
 * 19.1 and 19.5; "TileLang in practice: FlashAttention forward kernel",
 * sections 2.3-2.4 and 4.  The result is exact up to rounding: the only
 * precision drop is the bf16 rounding of the probabilities before the second
 * matrix product (ch.15 section 3.2; TileLang in practice section 4.5).
 *
 * Masks (ch.15 sections 3.4, 5.2, 5.3).  With off = Skv - Sq (queries are
 * aligned to the END of the keys, the KV-cache convention), key j is visible
 * to query i iff
 *     j < Skv
 *     and, if causal:              j <= i + off
 *     and, if window W > 0:        j > i + off - W   or   j < n_sink.
 * A query that sees no key gets O = +0.0 and LSE = -inf (ch.15 section
 * 5.1(2)).  The sliding window is only defined together with causal.
 *
 * Grouped-query attention (ch.15 section 4.8(1)): query head h reads
 * key/value head h / (Hq / Hkv); Hq must be a multiple of Hkv.
 *
 * Common rules for every entry point.
 *   - Pointers to tensors are DEVICE pointers owned by the caller, 16-byte
 *     aligned, to contiguous row-major tensors in the layouts stated below.
 *     The library never allocates or frees device memory; its only device
 *     state is a status word and the fixed scratch array of
 *     attn_decode_paged_noalloc.
 *   - Element types: q, k, v, o are bf16 (uint16 storage); lse is fp32.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream: they return after
 *     launching and never synchronise, except attn_device_status.
 *   - Return value: an attn_status code.  On any error nothing is launched.
 *     Errors found by a kernel (a bounded wait that ran out, an out-of-range
 *     page index) cannot be returned by the launching call; the kernel
 *     records them in a device-side status word read by attn_device_status.
 *   - Head dimension d: 64, 128 or 256 for every forward call (attn_fwd,
 *     attn_fwd_ex, attn_fwd_ex_sink, attn_fwd_strided, attn_fwd_paged; at
 *     d = 256 a CTA takes one 128-row query tile, with two score buffers and
 *     O in tensor memory), for the decode (at d = 256 the two consumer
 *     warps of a split each keep half of O) and for the backward (at
 *     d = 256 dV, dK and dQ come from three launches that stream 64-row
 *     tiles).  The device must be sm_103.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, Hq % Hkv != 0,
                               window without causal, workspace too small, ... */
  ATTN_ERR_UNSUPPORTED = 2, /* head dim not supported by the call, page size not 16, device not sm_103 */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_TIMEOUT = 4,     /* a kernel's bounded wait ran out (device status) */
  ATTN_ERR_BAD_INPUT = 5    /* a kernel met out-of-range device data, e.g. a page
                               index outside [0, num_pages_total) (device status) */
} attn_status;

/*
 * Dense attention forward, BSHD layout.
 *   q   [B, Sq,  Hq,  d]   bf16       k, v [B, Skv, Hkv, d]  bf16
 *   o   [B, Sq,  Hq,  d]   bf16 (out) lse  [B, Hq,  Sq]      fp32 (out, may be NULL)
 *   scale: multiplies Q K^T (1/sqrt(d) in the usual convention).
 *   causal: 0/1.  window: <= 0 for none, else W keys including the diagonal
 *   (requires causal).  No sink keys (see attn_fwd_ex).
 * Sizes: B, Hq, Hkv >= 1; Sq, Skv >= 0 (Sq == 0 or B == 0 launches nothing;
 * Skv == 0 writes O = 0, LSE = -inf).  q/k/v may be NULL only when their
 * tensor is empty.
 */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int Hq, int Hkv, int Sq, int Skv, int d,
                      float scale, int causal, int window, void* stream);

/*
 * Attention forward with sink keys and optional variable-length packing.
 *   cu_seqlens_q, cu_seqlens_k: NULL for the dense layout of attn_fwd (then
 *     B is the batch, max_Sq/max_Skv are Sq/Skv, total_q/total_k unused);
 *     otherwise DEVICE int32 arrays [B + 1] of prefix sums over B packed
 *     sequences (ch.15 section 5.3) and the layouts are
 *       q, o [total_q, Hq, d]   k, v [total_k, Hkv, d]   lse [Hq, total_q]
 *     with total_q = cu_seqlens_q[B], total_k = cu_seqlens_k[B] passed by
 *     the caller; max_Sq bounds every query length (it sizes the grid).
 *     Causal alignment is per sequence, to the end of its keys.
 *   n_sink: with a window, keys 0..n_sink-1 of each sequence stay visible
 *     to every query that may see them causally (n_sink > 0 needs window > 0).
 * Device-side checks: cu_seqlens entries that decrease or exceed the totals
 * are reported as ATTN_ERR_BAD_INPUT through attn_device_status and that
 * sequence is skipped.
 */
ATTN_API int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                         const int* cu_seqlens_q, const int* cu_seqlens_k,
                         int B, int Hq, int Hkv, int max_Sq, int max_Skv,
                         int total_q, int total_k, int d,
                         float scale, int causal, int window, int n_sink, void* stream);

/*
 * attn_fwd_ex with a logit sink per query head ("TileLang tutorial, ch.15
 * Operators: Attention", section 4.6, the attention-sink variant: the sink
 * adds one term to the softmax denominator).
 *   sink_logit: DEVICE fp32 array [Hq] (4-byte aligned), or NULL for none
 *     (then identical to attn_fwd_ex).  sink_logit[h] is a logit sigma_h in
 *     the units of scale * q.k (natural log) that joins every row of head h
 *     as one more softmax column with no value row:
 *       O_i   = sum_j e^(S_ij) V_j / (e^sigma_h + sum_j e^(S_ij))
 *       LSE_i = ln(e^sigma_h + sum_j e^(S_ij))       (j over visible keys)
 *     computed against max(sigma_h, max_j S_ij), so a large sigma does not
 *     overflow.  sigma_h = -inf means no sink for that head; +inf or NaN
 *     give undefined results.  A row that sees no key gets O = 0 and
 *     LSE = sigma_h.  The sink does not change which keys are visible; it
 *     combines freely with causal, window, n_sink (sink keys), GQA and
 *     varlen.
 * Other arguments, layouts and results are those of attn_fwd_ex.
 */
ATTN_API int attn_fwd_ex_sink(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k,
                              int B, int Hq, int Hkv, int max_Sq, int max_Skv,
                              int total_q, int total_k, int d,
                              float scale, int causal, int window, int n_sink,
                              const float* sink_logit, void* stream);

/*
 * Dense forward on tensors of any layout whose head dimension is contiguous,
 * e.g. BHSD ([B, H, S, d]) as well as BSHD ("TileLang tutorial, ch.15",
 * section 4.6: the two layouts differ only in index order; what matters is
 * that the copied dimension is contiguous).
 *   q_strides, k_strides, v_strides, o_strides: HOST arrays of three int64
 *     strides in elements, {batch, sequence row, head}, of q [B, Sq, Hq, d],
 *     k/v [B, Skv, Hkv, d] and o [B, Sq, Hq, d] indexed in that order; the d
 *     elements of a row are contiguous.  NULL means the contiguous BSHD
 *     strides of attn_fwd.  Every stride must be a positive multiple of 8
 *     elements (16 bytes); the tensor-map encoder may reject others
 *     (ATTN_ERR_INVALID_ARG).  o must not overlap itself or the inputs.
 *   lse stays [B, Hq, Sq] contiguous (may be NULL); sink_logit as in
 *   attn_fwd_ex_sink (may be NULL).  Other arguments as in attn_fwd_ex.
 */
ATTN_API int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int Sq, int Skv, int d,
                              const long long* q_strides, const long long* k_strides,
                              const long long* v_strides, const long long* o_strides,
                              float scale, int causal, int window, int n_sink,
                              const float* sink_logit, void* stream);

/*
 * Packed queries against a paged KV cache: chunked prefill, or several new
 * tokens per request (speculative decoding) ("TileLang tutorial, ch.15",
 * sections 3.4(2) and 5.3: the causal diagonal of a query block that ends at
 * the cache's end, past_len = keys - queries; section 4.6 for the paged
 * addressing of the decode variant, here with query blocks).
 *   q, o       [total_q, Hq, d] bf16, sequence b's queries at rows
 *              cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 (DEVICE int32 [B+1])
 *   lse        [Hq, total_q] fp32 (out, may be NULL)
 *   k_pages, v_pages [num_pages_total, page_size, Hkv, d] bf16 (page_size 16)
 *   page_table [B, max_pages_per_seq] int32, seqlens_k [B] int32 (DEVICE):
 *              sequence b's keys are its first seqlens_k[b] cache slots, slot
 *              t in physical page page_table[b][t / 16], row t % 16.
 *   causal: query i of sequence b (0-based in its block of Lq_b rows) sees
 *     keys j <= i + (seqlens_k[b] - Lq_b); rows with no key (Lq_b >
 *     seqlens_k[b]) get O = 0, LSE = -inf (or the sink).  window, n_sink and
 *     sink_logit (may be NULL) as in attn_fwd_ex / attn_fwd_ex_sink.
 *   Slots of a sequence's last page past seqlens_k[b] are read and given
 *   weight zero, so they must hold finite values.  Page-table entries past
 *   ceil(seqlens_k[b] / 16) are never read; an entry outside
 *   [0, num_pages_total) is not dereferenced: page 0 is read instead and
 *   ATTN_ERR_BAD_INPUT is set in the device status.  Sequence offsets that
 *   decrease, exceed total_q or max_Sq, or key counts above
 *   max_pages_per_seq * 16, likewise set ATTN_ERR_BAD_INPUT and that
 *   sequence is skipped.
 */
ATTN_API int attn_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int* page_table, const int* cu_seqlens_q, const int* seqlens_k,
                            void* o, float* lse, int B, int Hq, int Hkv, int max_Sq, int total_q,
                            int d, int page_size, int max_pages_per_seq, int num_pages_total,
                            float scale, int causal, int window, int n_sink,
                            const float* sink_logit, void* stream);

/*
 * Bytes of device workspace attn_bwd needs (two fp32 values per query row,
 * rows padded to multiples of 128).  0 on invalid sizes.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Sq);

/*
 * Backward pass of attn_fwd (dense BSHD, causal or not, GQA; attn_bwd_ex
 * adds sink keys, the window and packed sequences): from q, k, v, the
 * forward's o and lse and the
 * gradient dout of o, writes
 *   dq [B, Sq, Hq, d], dk, dv [B, Skv, Hkv, d]   (bf16, device, caller-owned)
 * with dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO, P = exp(scale Q K^T -
 * LSE) rebuilt from lse, dS = P (dO V^T - rowsum(dO * O)).  The pages give no
 * backward formulas; "TileLang tutorial, ch.15", section 5.4 reports the
 * error of a dQ accumulated atomically in bf16, which is why every gradient
 * here is accumulated in fp32 over its whole reduction by one CTA and
 * written once: results are bitwise repeatable.  dK and dV of a key head sum
 * over the Hq/Hkv query heads that read it.
 *   lse: the forward's [B, Hq, Sq] output (rows with -inf, which saw no key,
 *   get dq = 0 and contribute nothing).  workspace: device buffer of at least
 *   attn_bwd_workspace_size(B, Hq, Sq) bytes, overwritten.  Sq == 0 zeroes
 *   dk and dv; Skv == 0 zeroes dq.  d must be 64, 128 or 256.
 * The gradient kernels may overlap one another on the stream (each starts
 * on the SMs the one before it frees); work queued on the stream after the
 * call still starts only once all three gradients are written.
 */
ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      int B, int Hq, int Hkv, int Sq, int Skv, int d, float scale, int causal,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass of attn_fwd_ex: the gradients of attn_bwd, with the same
 * masks as the forward (sink keys, sliding window, packed sequences;
 * "TileLang tutorial, ch.15", sections 3.4, 5.2 and 5.3).
 *   cu_seqlens_q, cu_seqlens_k: NULL for the dense layout of attn_bwd; else
 *   int32 [B + 1] offsets of B packed sequences as in attn_fwd_ex, with q, o,
 *   dout, dq [total_q, Hq, d], k, v, dk, dv [total_k, Hkv, d] and lse
 *   [Hq, total_q]; max_Sq / max_Skv bound every sequence's lengths (the dense
 *   sizes when not packed).  A packed sequence with offsets out of range is
 *   left out and reported as ATTN_ERR_BAD_INPUT (attn_device_status).
 *   window, n_sink: as in attn_fwd_ex (window > 0 requires causal, n_sink > 0
 *   requires a window).
 *   workspace: at least attn_bwd_workspace_size(B, Hq, max_Sq) bytes.
 *   Keys no query sees get dk = dv = 0; queries that see no key get dq = 0.
 * Errors as attn_bwd.
 */
ATTN_API int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                         int Hkv, int max_Sq, int max_Skv, int total_q, int total_k, int d,
                         float scale, int causal, int window, int n_sink, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Backward pass of attn_fwd_ex_sink: attn_bwd_ex's gradients plus that of
 * the logit sink ("TileLang tutorial, ch.15", section 4.6, the sink as one
 * more softmax column without a value row).
 *   lse: the forward's LSE, which includes the sink term; with it the
 *   dq, dk, dv of attn_bwd_ex are those of the sink-augmented softmax.
 *   sink_logit: DEVICE fp32 [Hq], the forward's sigma (-inf: none).
 *   dsink: DEVICE fp32 [Hq] (out): dL/dsigma_h = -sum over the rows of head h
 *     (every sequence) of P_sink * rowsum(dO * O), P_sink = e^(sigma_h - LSE).
 *     Each head is summed by one block in a fixed order, so repeated calls
 *     give identical bits.  No query: dsink = 0.
 * Both sink pointers must be set (ATTN_ERR_INVALID_ARG otherwise); the other
 * arguments and errors are those of attn_bwd_ex.
 */
ATTN_API int attn_bwd_ex_sink(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int max_Sq, int max_Skv, int total_q, int total_k, int d,
                              float scale, int causal, int window, int n_sink,
                              const float* sink_logit, float* dsink, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace attn_decode_paged needs for these sizes (split
 * partial outputs and log-sum-exps, fp32, and the batch's requests ordered
 * longest first, int32 [B]).  0 on invalid sizes.
 */
ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * One-token decode over a paged KV cache, split-KV with a log-sum-exp merge
 * ("TileLang tutorial, ch.15", sections 4.6 and 4.8(2)-(3), 5.4;
 * "learn-cuda-from-scratch, ch.12 FlashAttention", section 12.9.4).
 *   q        [B, Hq, d] bf16              o   [B, Hq, d] bf16 (out)
 *   lse      [B, Hq] fp32 (out, may be NULL)
 *   k_pages, v_pages [num_pages_total, page_size, Hkv, d] bf16
 *   page_table [B, max_pages_per_seq] int32: logical page p of request b is
 *     physical page page_table[b*max_pages_per_seq + p]; entries at or past
 *     ceil(seqlens[b] / page_size) are never read.
 *   seqlens  [B] int32, 0 <= seqlens[b] <= max_pages_per_seq * page_size.
 *   Request b's query sees its first seqlens[b] keys.  A request with no key
 *   gets O = 0, LSE = -inf.
 *   num_splits (1..64): the keys of each request are cut at page granularity,
 *   pps = ceil(npages_b / num_splits) pages per split; the partial results
 *   are merged in ascending split order, so repeated calls give identical
 *   bits.
 *   workspace: device buffer of at least attn_decode_workspace_size(...)
 *   bytes, no initial contents required; it is overwritten by every call, so
 *   calls sharing one workspace must not overlap in time.
 * page_size must be 16.  Out-of-range page indices are not dereferenced:
 * they read as zero keys and set ATTN_ERR_BAD_INPUT in the device status.
 */
ATTN_API int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                               const int* page_table, const int* seqlens, void* o, float* lse,
                               int B, int Hq, int Hkv, int d, int page_size,
                               int max_pages_per_seq, int num_pages_total, int num_splits,
                               float scale, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * attn_decode_paged with a logit sink per query head (section 4.6 as for
 * attn_fwd_ex_sink): sink_logit is a DEVICE fp32 array [Hq] or NULL.  The
 * sink joins the merge of the split partials as one more denominator term
 * with no output, M = max(sigma_h, lse_s):
 *   O = sum_s e^(lse_s - M) O_s / (e^(sigma_h - M) + sum_s e^(lse_s - M)),
 *   LSE = M + ln(e^(sigma_h - M) + sum_s e^(lse_s - M)),
 * summed in ascending split order after the sink term.  A request with no
 * key gets O = 0 and LSE = sigma_h.  Other arguments are those of
 * attn_decode_paged.
 */
ATTN_API int attn_decode_paged_sink(const void* q, const void* k_pages, const void* v_pages,
                                    const int* page_table, const int* seqlens, void* o,
                                    float* lse, int B, int Hq, int Hkv, int d, int page_size,
                                    int max_pages_per_seq, int num_pages_total, int num_splits,
                                    float scale, const float* sink_logit, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * attn_decode_paged without a workspace argument: the same decode, for
 * callers that cannot allocate device memory themselves (a serving loop that
 * must not allocate once it is running, a host program whose plugins may only
 * use memory handed to them, code that cannot afford the device-wide
 * synchronisation an allocation may cause).  There is no counterpart on the
 * source pages: it is an addition of this library.
 *   The split partials go to one scratch array built into the library
 *   (16 MiB, held on every device that loads the library until the process
 *   exits).  Calls needing more than that (attn_decode_workspace_size(...)
 *   > 16 MiB) return ATTN_ERR_INVALID_ARG and launch nothing.  The library
 *   allocates nothing on this path.
 *   The first call on a device looks up the scratch array's device address
 *   (with that device current) and keeps it; make that first call before
 *   any stream capture.
 *   Every call on a device shares the one scratch array and leaves its last
 *   contents there (nothing in it needs to start at zero), so calls whose
 *   executions overlap on the GPU race with each other: issue them on one
 *   stream, or order them.
 * Arguments, layouts and results are those of attn_decode_paged.
 */
ATTN_API int attn_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                       const int* page_table, const int* seqlens, void* o,
                                       float* lse, int B, int Hq, int Hkv, int d, int page_size,
                                       int max_pages_per_seq, int num_pages_total, int num_splits,
                                       float scale, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device-side status word
 * of the current device (ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_BAD_INPUT, or
 * ATTN_ERR_UNSUPPORTED when a kernel found its dynamic shared memory off the
 * 1024-byte boundary its layout assumes and wrote nothing), or ATTN_ERR_CUDA
 * if the synchronisation itself failed.
 */
ATTN_API int attn_device_status(void* stream);

/*
 * Launches a one-warp kernel whose bounded wait (the same helper every
 * kernel of the library uses) waits on a barrier that nothing completes,
 * with a limit of `limit_us` microseconds (1..1000000).  The kernel returns
 * cleanly and the next attn_device_status reports ATTN_ERR_TIMEOUT.  Used to
 * test failure reporting without faulting or hanging the GPU.
 */
ATTN_API int attn_check_wait_timeout(int limit_us, void* stream);

/* Static English text for a status code. */
ATTN_API const char* attn_status_string(int status);

/* Text of the last ATTN_ERR_CUDA / argument error seen by this thread. */
ATTN_API const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
