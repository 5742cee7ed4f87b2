/*
 * libattn -- exact scaled dot-product attention for NVIDIA GB300 (sm_103a).
 *
 * What is computed (every entry point below), for batch b, query head h and
 * KV head kv = h / (hq / hkv)  (GQA: contiguous groups of query heads share
 * one KV head):
 *
 *   s_ij = scale * <q_i, k_j>                       "FlashAttention完整说明" §一
 *   s_ij = softcap * tanh(s_ij / softcap)  if softcap > 0, applied BEFORE the
 *          mask (Inference Cookbook FAQ Q22)
 *   mask: query i sits at key position p_i = i + (sk - sq)  (bottom-right
 *          alignment, Inference Cookbook FAQ Q6) and sees key j iff
 *          p_i - win_l <= j <= p_i + win_r   (FAQ Q21; -1 = unbounded side;
 *          causal != 0 forces win_r = 0)
 *   P = softmax over the visible keys, O = P V,  LSE_i = m_i + ln(l_i)
 *          (the saved softmax statistics of "FlashAttention完整说明" §二.2)
 *
 * scale must be finite and >= 0 (the FlashAttention default is 1/sqrt(d),
 * Inference Cookbook FAQ Q12); softcap <= 0 turns the cap off.
 *
 * Rows with no visible key produce O = 0 and LSE = -inf and get zero
 * gradient.  The score matrix is never written to memory: the kernels tile
 * Q/K/V through shared memory and use an online softmax (§二.1), and the
 * backward recomputes S and P from Q, K and the saved LSE (§二.2).
 *
 * Layout (Inference Cookbook FAQ Q5): q/out/dout/dq are (batch, seqlen_q,
 * hq, d), k/v/dk/dv are (batch, seqlen_k, hkv, d), all contiguous, element
 * type fp16 or bf16 (dtype below; "FlashAttention完整说明" §八: FP16/BF16
 * only).  d must be 64, 128 or 256.  LSE is fp32 (batch, hq, seqlen_q); for
 * the varlen calls it is (hq, total_q).  Accumulation is fp32; outputs are
 * rounded to the element type with round-to-nearest-even.
 *
 * Ownership and streams: every pointer is a DEVICE pointer owned by the
 * caller, except where noted.  The library allocates nothing and never
 * synchronises the stream on these calls; scratch memory is a caller-owned
 * `workspace` sized by the matching *_workspace_size query.  All work is
 * enqueued on `stream` (NULL = the legacy default stream), so a call can be
 * captured into a CUDA graph when its pointers stay fixed (Inference Cookbook
 * FAQ Q19).
 *
 * Errors: arguments are validated on the host before anything is enqueued;
 * an invalid call returns a nonzero status and launches nothing.  A launch
 * failure returns ATTN_ERR_CUDA.  Data-dependent faults detected on the
 * device (a block_table entry outside the page pool, a varlen length above the
 * stated maximum, a bounded wait that timed out) skip the offending work and
 * raise a sticky device error word, read and cleared by
 * attn_get_device_error().
 */
#ifndef LIBATTN_H
#define LIBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = 1,     /* bad pointer, size or flag combination          */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request this build does not implement    */
  ATTN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required     */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed  */
  ATTN_ERR_TIMEOUT = 5,     /* a device-side bounded wait expired             */
  ATTN_ERR_DEVICE = 6       /* device-side data check failed (see above)      */
} attn_status;

enum { ATTN_F16 = 0, ATTN_BF16 = 1 };

/* Library version string, e.g. "libattn 0.1.0 (sm_103a)".  Host only. */
const char *attn_version(void);

/* Human-readable name of a status code.  Host only. */
const char *attn_status_str(attn_status s);

/*
 * Dense forward.  q (b,sq,hq,d), k/v (b,sk,hkv,d), out (b,sq,hq,d) in dtype;
 * lse (b,hq,sq) fp32, required (the backward reads it).  sq == 0 or sk == 0
 * is valid (sk == 0: every row is empty).  hq % hkv must be 0.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                     int dtype, int b, int sq, int sk, int hq, int hkv, int d, float scale,
                     int causal, int win_l, int win_r, float softcap, attn_stream_t stream);

/*
 * Backward ("FlashAttention完整说明" §二.2: recompute S and P from Q, K and
 * the saved LSE).  Inputs q, k, v, out, lse as produced by attn_fwd with the
 * same arguments, dout (b,sq,hq,d).  Outputs dq (b,sq,hq,d), dk/dv
 * (b,sk,hkv,d) in dtype, fully overwritten.
 *
 * deterministic != 0 makes dq bitwise reproducible run to run (no
 * floating-point atomics, Inference Cookbook FAQ Q11); deterministic == 0
 * may accumulate dq with fp32 atomics in an unspecified order.
 *
 * workspace: device scratch of at least attn_bwd_workspace_size(...) bytes,
 * 256-byte aligned; its contents need not be initialised.
 */
size_t attn_bwd_workspace_size(int b, int sq, int sk, int hq, int hkv, int d, int deterministic);

attn_status attn_bwd(const void *q, const void *k, const void *v, const void *out,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv,
                     int dtype, int b, int sq, int sk, int hq, int hkv, int d, float scale,
                     int causal, int win_l, int win_r, float softcap, int deterministic,
                     void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd / attn_bwd for inputs (and, in the backward, gradients) whose
 * tokens are not densely packed: *_row_stride is the number of elements from
 * token r to token r + 1 of that tensor (row r = batch * s + position; head
 * h of a row starts h * d elements after the row; batch entries follow each
 * other at s rows).  0 means contiguous (heads * d).  This takes the packed
 * layouts without copies -- qkv (b, s, 3, hq, d) of the qkvpacked call
 * ("flash_attn FlashAttention完整说明" §六.1): q = qkv, k = qkv + hq*d,
 * v = qkv + 2*hq*d, every stride 3*hq*d; kv (b, s, 2, hkv, d) of the
 * kvpacked call (Inference Cookbook FAQ Q7): k = kv, v = kv + hkv*d, both
 * strides 2*hkv*d -- and writes the gradients into the same packed layout.
 * out, lse and dout stay contiguous.  A non-zero stride must be at least
 * heads * d and a multiple of 8 (16-byte rows); every pointer 16-byte
 * aligned; otherwise ATTN_ERR_INVALID.  Everything else as attn_fwd /
 * attn_bwd.
 *
 * pack_gqa (forward; Inference Cookbook FAQ Q15): with GQA, the g = hq/hkv
 * query heads of a KV head may share each 128-row tile (128/g positions x g
 * heads), so short query sequences do not leave tiles empty and each K/V
 * tile serves g heads.  < 0: automatic (on when sq <= 128 and g divides 128,
 * which is what attn_fwd and attn_fwd_varlen use); 0: off; > 0: on, and
 * ATTN_ERR_UNSUPPORTED when g does not divide 128.  The result does not
 * depend on the choice.
 */
attn_status attn_fwd_strided(const void *q, const void *k, const void *v, void *out, float *lse,
                             int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride,
                             int dtype, int b, int sq, int sk, int hq, int hkv, int d,
                             float scale, int causal, int win_l, int win_r, float softcap,
                             int pack_gqa, attn_stream_t stream);

attn_status attn_bwd_strided(const void *q, const void *k, const void *v, const void *out,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride,
                             int64_t dq_row_stride, int64_t dk_row_stride,
                             int64_t dv_row_stride, int dtype, int b, int sq, int sk, int hq,
                             int hkv, int d, float scale, int causal, int win_l, int win_r,
                             float softcap, int deterministic, void *workspace,
                             size_t workspace_bytes, attn_stream_t stream);

/*
 * Varlen (packed) forward, Inference Cookbook FAQ Q8.  q (total_q,hq,d),
 * k/v (total_k,hkv,d), out (total_q,hq,d); lse (hq,total_q) fp32.
 * cu_seqlens_q/k: DEVICE int32 arrays of batch+1 offsets starting at 0.
 * Sequence i has sq_i = cu_q[i+1]-cu_q[i] queries and sk_i keys; its masks
 * align bottom-right within the sequence.  max_seqlen_q/k must bound every
 * sq_i/sk_i (a sequence that exceeds them is skipped and raises the device
 * error word); total_q/total_k must equal cu_q[batch]/cu_k[batch].
 */
attn_status attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, int dtype, int hq, int hkv, int d, float scale,
                            int causal, int win_l, int win_r, float softcap,
                            attn_stream_t stream);

size_t attn_bwd_varlen_workspace_size(int batch, int max_seqlen_q, int max_seqlen_k,
                                      int total_q, int total_k, int hq, int hkv, int d,
                                      int deterministic);

attn_status attn_bwd_varlen(const void *q, const void *k, const void *v, const void *out,
                            const float *lse, const void *dout, void *dq, void *dk, void *dv,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, int dtype, int hq, int hkv, int d, float scale,
                            int causal, int win_l, int win_r, float softcap, int deterministic,
                            void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * Decode against a KV cache, with optional append (Inference Cookbook FAQ
 * Q17, Q18, Q14).
 *
 * Paged (block_table != NULL): k_cache/v_cache are a page pool
 * (num_pages, page_size, hkv, d); logical position t of batch entry i lives
 * in page block_table[i*max_pages_per_seq + t/page_size], slot t%page_size.
 * page_size must be a multiple of 128.  Contiguous (block_table == NULL):
 * k_cache/v_cache are (b, page_size, hkv, d) -- one "page" of page_size
 * tokens per batch entry; pass num_pages = b and max_pages_per_seq = 1.
 *
 * cache_seqlens (b) int32 DEVICE array: tokens already in the cache.  It is
 * read, never written: the caller advances it by s_new after the call (FAQ
 * Q17).  k_new/v_new (b, s_new, hkv, d), or NULL with s_new = 0: rows written
 * into the cache at positions cache_seqlens[i] .. cache_seqlens[i]+s_new-1,
 * and attended to.  Batch entry i attends over L_i = cache_seqlens[i] + s_new
 * keys with the bottom-right mask (query r sits at position L_i - sq + r).
 * Every L_i must fit max_pages_per_seq * page_size; the block_table entries
 * used must lie in [0, num_pages) (checked on the device: the device error
 * word is raised, and a split that meets a bad entry contributes the empty
 * result -- O = 0, LSE = -inf -- so the output is deterministic but not
 * meaningful for that batch entry).
 *
 * q (b,sq,hq,d), out (b,sq,hq,d), lse (b,hq,sq) fp32.
 *
 * num_splits: 0 = choose from the SM count and the cache length (FAQ Q14),
 * else the number of key ranges each (batch, KV head) is split into; the
 * split results are merged by their LSE.  workspace: at least
 * attn_kvcache_workspace_size(...) bytes (may be 0 when one split is used).
 */
int attn_kvcache_num_splits(int b, int sq, int hq, int hkv, int d, int max_seqlen_k,
                            int num_splits);

size_t attn_kvcache_workspace_size(int b, int sq, int hq, int hkv, int d, int max_seqlen_k,
                                   int num_splits);

attn_status attn_fwd_kvcache(const void *q, void *k_cache, void *v_cache, const void *k_new,
                             const void *v_new, const int32_t *cache_seqlens,
                             const int32_t *block_table, int num_pages, int page_size,
                             int max_pages_per_seq, void *out, float *lse, int dtype, int b,
                             int sq, int s_new, int hq, int hkv, int d, float scale, int causal,
                             int win_l, int win_r, float softcap, int num_splits,
                             void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd_kvcache_noalloc -- the decode of attn_fwd_kvcache for callers
 * that cannot allocate device memory.  The pages have no counterpart; it
 * exists for hosts such as code that runs while a CUDA graph is being
 * captured (cudaMalloc cannot be captured), inference-server plugins whose
 * device memory belongs to a pool they may not grow, and plain C callers
 * without a CUDA allocator.  Arguments and results are those of
 * attn_fwd_kvcache without `workspace`: the split partials go to a 32 MiB
 * array inside the library (held on every GPU that loads the library until
 * the process exits).  A call whose attn_kvcache_workspace_size(...) exceeds
 * 32 MiB returns ATTN_ERR_WORKSPACE and launches nothing.  Nothing is
 * allocated or freed.  The first call on a device looks up the array's
 * device address (a host-side query, once per device); make that first call
 * before any stream capture.  All calls share the one array: calls that
 * overlap on the GPU (different streams, or several threads) race on it and
 * must be serialised by the caller.
 */
attn_status attn_fwd_kvcache_noalloc(const void *q, void *k_cache, void *v_cache,
                                     const void *k_new, const void *v_new,
                                     const int32_t *cache_seqlens, const int32_t *block_table,
                                     int num_pages, int page_size, int max_pages_per_seq,
                                     void *out, float *lse, int dtype, int b, int sq, int s_new,
                                     int hq, int hkv, int d, float scale, int causal, int win_l,
                                     int win_r, float softcap, int num_splits,
                                     attn_stream_t stream);

/*
 * FP8 forward (Inference Cookbook FAQ Q20: FP8 inside, BF16 out; FAQ Q10
 * gives 1e-2 absolute / 1e-2 relative as the FP8 tolerance).  q (b,sq,hq,d)
 * and k, v (b,sk,hkv,d) hold OCP FP8 E4M3 bytes; the inputs they stand for
 * are q * descale_q, k * descale_k and v * descale_v (per-tensor factors,
 * finite and > 0).  S = Q K^T runs on the tensor cores in FP8 with fp32
 * accumulation; V is widened to bf16 into `workspace` (exactly) and P V runs
 * in bf16.  out (b,sq,hq,d) is bf16 and lse (b,hq,sq) fp32, as attn_fwd.
 * Masks, softcap, GQA as attn_fwd.  d must be 128 and sk > 0, else
 * ATTN_ERR_UNSUPPORTED.  workspace: attn_fwd_fp8_workspace_size(...) bytes,
 * 256-byte aligned.
 */
size_t attn_fwd_fp8_workspace_size(int b, int sk, int hkv, int d);

attn_status attn_fwd_fp8(const void *q, const void *k, const void *v, void *out, float *lse,
                         float descale_q, float descale_k, float descale_v, int b, int sq, int sk,
                         int hq, int hkv, int d, float scale, int causal, int win_l, int win_r,
                         float softcap, void *workspace, size_t workspace_bytes,
                         attn_stream_t stream);

/*
 * Debug only: the attention probabilities of a forward call (Inference
 * Cookbook FAQ Q9, return_attn_probs: the whole (batch, heads, seqlen_q,
 * seqlen_k) matrix costs O(N^2) memory, so it is for tests and debugging,
 * never the hot path).  q (b,sq,hq,d), k (b,sk,hkv,d) in dtype and lse
 * (b,hq,sq) fp32 as attn_fwd produced it for the same arguments.  p
 * (b,hq,sq,sk) fp32 is fully overwritten: P_ij = exp(s_ij - LSE_i) for every
 * visible (i, j), 0 elsewhere, with s the scaled (and soft-capped) score of
 * attn_fwd, so each non-empty row sums to 1 and rows that see no key are 0.
 * Same argument checks as attn_fwd; p must be 16-byte aligned.
 */
attn_status attn_fwd_probs(const void *q, const void *k, const float *lse, float *p, int dtype,
                           int b, int sq, int sk, int hq, int hkv, int d, float scale,
                           int causal, int win_l, int win_r, float softcap,
                           attn_stream_t stream);

/*
 * cache_seqlens[i] += s_new for i in [0, b), as one kernel on `stream`.
 * attn_fwd_kvcache appends k_new/v_new but never advances the lengths; the
 * caller does (Inference Cookbook FAQ Q17).  Done on the device, the
 * advance lets a whole decode step -- attn_fwd_kvcache then this call -- be
 * captured once in a CUDA graph and replayed with fixed addresses (FAQ
 * Q19).  cache_seqlens: device int32[b], 4-byte aligned.  b == 0 is a no-op;
 * b < 0, s_new < 0 or a NULL array with b > 0 is ATTN_ERR_INVALID.
 */
attn_status attn_kvcache_advance(int32_t *cache_seqlens, int b, int s_new, attn_stream_t stream);

/*
 * Reads and clears the sticky device error word of the current device
 * (synchronises `stream`; diagnostic use, not for the hot path).  Returns
 * ATTN_OK, ATTN_ERR_DEVICE or ATTN_ERR_TIMEOUT.  If `detail` is not NULL it
 * receives the raw error word (which check fired).
 */
attn_status attn_get_device_error(attn_stream_t stream, int *detail);

/*
 * Number of kernels this library has enqueued since it was loaded (all
 * devices and threads; a relaxed atomic counter).  Lets a caller count the
 * library's launches inside a timed region.  Host only.
 */
unsigned long long attn_launch_count(void);

/*
 * Sets the wall-clock limit (nanoseconds) of every device-side wait of the
 * calls that follow (all devices, all threads); 0 restores the default of
 * 2 s.  Returns the previous limit.  Host only; the limit is read when a call
 * is made, so it does not change work already enqueued.  A wait that reaches
 * the limit gives up, its kernel skips the rest of its work, and the call's
 * outputs are unspecified; attn_get_device_error() then reports
 * ATTN_ERR_TIMEOUT.  Meant for tests of that error path: a very small limit
 * makes ordinary waits expire.  (The library's own guard against a kernel
 * that never finishes, not a counterpart of anything on the pages.)
 */
unsigned long long attn_set_wait_limit_ns(unsigned long long ns);

/*
 * Test hook for that error path (not for production use): while `on` is
 * non-zero, the tensor-core kernels of the calls that follow make their MMA
 * issuer first wait on a barrier that nothing completes, so that wait runs
 * out after the wait limit, the kernel abandons its work (draining its own
 * copies and MMAs first) and the call's outputs are unspecified;
 * attn_get_device_error() then reports ATTN_ERR_TIMEOUT.  Kernels on the
 * CUDA cores do not wait and are unaffected.  Returns the previous setting.
 * Host only; read when a call is made.
 */
int attn_set_test_stall(int on);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_H */
