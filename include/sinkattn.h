/*
 * sinkattn — grouped-query attention with a learned per-head softmax sink,
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation ("GPT-OSS on Day 0", Perplexity, section "Kernels for GPT-OSS /
 * Sink attention"; "Attention: GQA with attention sinks"):
 *
 *     attn = softmax(q @ k^T * sm_scale + sink) * V
 *
 * where the sink s_h of query head h is one extra logit column whose value row
 * is zero:
 *
 *     out_i = sum_j e^{l_j - M} v_j / (e^{s_h - M} + sum_j e^{l_j - M}),
 *     l_j   = sm_scale * q_i . k_j,   M = max(s_h, max_j l_j),
 *     lse_i = M + ln(e^{s_h - M} + sum_j e^{l_j - M})      (natural log, sink included).
 *
 * Several query heads share one KV head (GQA): query head h reads KV head
 * floor(h / G), G = num_qo_heads / num_kv_heads. The online softmax seeds its
 * running max with the head's sink (m = s_h, d = 1), so the sink is counted
 * exactly once; when the keys are split into chunks (split-KV decode), the
 * chunks carry no sink and the merge seeds with it (same section: the sink
 * belongs to one block only).
 *
 * Layouts (all device memory, row-major, contiguous):
 *   q, out       bf16 [total_q, Hq, d]  (token-major). Decode: total_q = batch*q_len,
 *                token b*q_len + t is draft t of sequence b.
 *   k, v         bf16 ragged HND ("Hosting Qwen on Blackwell", section "Deployment on
 *                GB200 NVL72": heads leading, tokens contiguous): sequence b is the
 *                contiguous block [Hkv, Lk_b, d] starting at element Hkv*cu_k[b]*d.
 *   sinks        fp32 [Hq], natural-log units of the scaled logits; NULL = no sink.
 *   lse          fp32 [total_q, Hq]; NULL = not written.
 *   cu_seqlens_* int32 [batch+1], non-decreasing, cu[0] = 0 (device memory).
 *
 * Masking: query i of a sequence with Lq queries and Lk keys sits at position
 * p = Lk - Lq + i (queries are the last Lq positions). causal: key j visible
 * iff j <= p. window W > 0 (requires causal): additionally j > p - W, i.e. the
 * W keys p-W+1 .. p. A row with no visible key and no sink gets out = 0,
 * lse = -inf; with a sink and no key, out = 0, lse = s_h.
 *
 * Supported: head_dim 64 or 128; num_qo_heads % num_kv_heads == 0; sm_scale > 0.
 *
 * Ownership and streams: the caller allocates and owns every buffer,
 * including the decode workspace. The library never allocates, frees or
 * synchronises in these calls; it enqueues kernels on `stream` (a
 * cudaStream_t; NULL = legacy default stream) and returns. Inputs are read
 * only. q, k, v, out and the partial buffers must be 16-byte aligned.
 *
 * Errors: every call validates its arguments on the host before launching
 * anything and returns a status code; on error nothing is launched and
 * sinkattn_last_error() (thread-local) describes the problem. Faults inside a
 * kernel (for example a bounded wait that gave up, or device-side lengths
 * that contradict the host-side sizes) are recorded in a device status word
 * that sinkattn_debug_status() reads.
 */
#ifndef SINKATTN_H_
#define SINKATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SINKATTN_API __attribute__((visibility("default")))
#else
#define SINKATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum sinkattn_status {
  SINKATTN_OK = 0,
  SINKATTN_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad workspace */
  SINKATTN_UNSUPPORTED = 2,  /* head_dim not 64/128, Hq % Hkv != 0, window without causal */
  SINKATTN_CUDA_ERROR = 3,   /* a CUDA runtime/driver call or launch failed */
  SINKATTN_TIMEOUT = 4,      /* device status: a bounded wait inside a kernel gave up */
  SINKATTN_BAD_LENGTHS = 5   /* device status: cu_seqlens/kv_indptr contradict the host sizes */
};

/*
 * Prefill / varlen attention with sink, single pass (no split), output
 * normalised. Steps: logits, mask, online softmax seeded with the sink,
 * P·V, finalize ("GPT-OSS on Day 0", "Kernels for GPT-OSS / Sink attention").
 *
 *   q [total_q, Hq, d], k/v ragged HND, sinks [Hq] or NULL,
 *   cu_seqlens_q / cu_seqlens_k [batch+1] (device),
 *   batch, total_q, max_seqlen_q, max_seqlen_k: host-side sizes for the grid
 *     (max_seqlen_* must bound every sequence; total_q = cu_seqlens_q[batch]),
 *   causal (0/1), window (<= 0: none; > 0 requires causal),
 *   out [total_q, Hq, d] bf16, lse [total_q, Hq] fp32 or NULL.
 * Each sequence needs Lq_b <= Lk_b.
 */
SINKATTN_API int sinkattn_prefill(const void* q, const void* k, const void* v, const float* sinks,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                     int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k,
                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                     float sm_scale, int32_t causal, int32_t window, void* out, float* lse,
                     void* stream);

/*
 * Split-KV decode / MTP, step 1: per-chunk partial state WITHOUT the sink
 * (heads and KV length both parallel: same section, "parallelise over heads
 * and KV sequence length").
 *
 *   q [batch*q_len, Hq, d] bf16; k/v ragged HND with kv_indptr [batch+1] (device);
 *   max_kv_len bounds every Lk_b (host); each sequence needs Lk_b >= q_len.
 *   Sequence b's keys are cut into num_splits chunks of
 *   c = 64 * ceil(Lk_b / (64 * num_splits)) keys (ceil(Lk_b / num_splits)
 *   rounded up to whole 64-key tiles); chunk s covers
 *   [s*c, min((s+1)*c, Lk_b)) and may be empty.
 *   part_md:  fp32 [batch*q_len, Hq, num_splits, 2]: (m_s, d_s), natural
 *             units, with m_s + ln d_s = ln sum_j e^{l_j}, the chunk's
 *             log-sum-exp over its visible keys;
 *   part_acc: fp32 [batch*q_len, Hq, num_splits, d]: d_s times the chunk's
 *             softmax-weighted mean of v_j, i.e. sum_j e^{l_j - m_s} v_j.
 *   The pair is defined up to the common rescale (m_s + c, d_s e^{-c},
 *   acc e^{-c}), which the merge is invariant to. The warp-level kernel
 *   writes m_s = the chunk's largest visible logit and d_s = the exact sum;
 *   the tcgen05 kernel writes d_s = the sum of the bf16-rounded weights its
 *   P.V product applied, with m_s adjusted so that m_s + ln d_s stays exact.
 *   An empty chunk gives (-inf, 0) and acc 0.
 */
SINKATTN_API int sinkattn_decode_split(const void* q, const void* k, const void* v,
                          const int32_t* kv_indptr, int32_t batch, int32_t q_len,
                          int32_t max_kv_len, int32_t num_qo_heads, int32_t num_kv_heads,
                          int32_t head_dim, float sm_scale, int32_t causal, int32_t window,
                          int32_t num_splits, float* part_acc, float* part_md, void* stream);

/*
 * Split-KV decode / MTP, step 2: fold the num_splits partials of every
 * (row, head) with the sink counted exactly once: the running state starts at
 * m = s_h, d = 1 (m = -inf, d = 0 without a sink) and absorbs each chunk with
 * the rescale to the larger maximum; out = acc / d, lse = m + ln d ("GPT-OSS
 * on Day 0", section "Kernels for GPT-OSS / Sink attention": the running max
 * m and scale d of the online softmax, the max seeded with the sink and d
 * with 1, the sink in the first block only when the sequence is split).
 *   part_acc/part_md as produced by sinkattn_decode_split; rows = batch*q_len;
 *   out [rows, Hq, d] bf16; lse [rows, Hq] fp32 or NULL.
 */
SINKATTN_API int sinkattn_merge(const float* part_acc, const float* part_md, const float* sinks,
                   int32_t rows, int32_t num_qo_heads, int32_t head_dim, int32_t num_splits,
                   void* out, float* lse, void* stream);

/*
 * Split-KV decode / MTP in one call ("GPT-OSS on Day 0", section "Kernels for
 * GPT-OSS / Sink attention": parallel over heads and KV length, the sink
 * counted once; "Hosting Qwen on Blackwell", section "Decoders": MTP drafts,
 * q_len > 1, attend causally to the cache): sinkattn_decode_split then
 * sinkattn_merge on the same stream, with the partials in the caller's workspace (at least
 * sinkattn_decode_workspace_bytes() bytes, 256-byte aligned, device memory;
 * contents on entry do not matter). num_splits <= 0 selects
 * sinkattn_decode_default_splits(). When a KV head has more query rows than
 * one 128-row tile (G x q_len > 128, e.g. 16 drafts of 16 heads) and the
 * kernel choice is SINKATTN_DECODE_AUTO, the call runs the single-pass
 * prefill kernel instead (the drafts are its queries, bottom-right causal,
 * every KV tile read once); the workspace is then unused and num_splits has
 * no effect on the result.
 */
SINKATTN_API int sinkattn_decode(const void* q, const void* k, const void* v, const int32_t* kv_indptr,
                    int32_t batch, int32_t q_len, int32_t max_kv_len, int32_t num_qo_heads,
                    int32_t num_kv_heads, int32_t head_dim, float sm_scale, int32_t causal,
                    int32_t window, int32_t num_splits, const float* sinks, void* workspace,
                    size_t workspace_bytes, void* out, float* lse, void* stream);

/*
 * Split-KV decode / MTP with the merge done on chip (no workspace): the
 * num_splits chunks of one (sequence, KV head) run as one thread-block
 * cluster; each chunk's partial (m, d, acc) stays in its CTA's shared memory
 * and the cluster folds them through distributed shared memory, seeding the
 * running state with the sink so it counts exactly once ("GPT-OSS on Day 0",
 * section "Kernels for GPT-OSS / Sink attention": parallel over heads and KV
 * length, the sink in one block only). Same chunking and results as
 * sinkattn_decode_split followed by sinkattn_merge.
 *   Arguments as sinkattn_decode without the workspace; num_splits <= 0
 *   selects sinkattn_decode_default_splits(); 1 <= num_splits <= 16 (a
 *   cluster of more than 16 CTAs is not launched: SINKATTN_UNSUPPORTED).
 *   out [batch*q_len, Hq, d] bf16; lse [batch*q_len, Hq] fp32 or NULL.
 */
SINKATTN_API int sinkattn_decode_fused(const void* q, const void* k, const void* v,
                                       const int32_t* kv_indptr, int32_t batch, int32_t q_len,
                                       int32_t max_kv_len, int32_t num_qo_heads,
                                       int32_t num_kv_heads, int32_t head_dim, float sm_scale,
                                       int32_t causal, int32_t window, int32_t num_splits,
                                       const float* sinks, void* out, float* lse, void* stream);

/*
 * sinkattn_decode for callers that cannot allocate device memory (for example
 * code inside another runtime whose memory manager owns all device memory and
 * gives plugins no allocator, or loops where a cudaMalloc, which may
 * synchronise the device, is not acceptable). The pages have no counterpart:
 * this is a deployment convenience, not part of the method.
 *
 * Same arguments and results as sinkattn_decode minus the workspace: the
 * partials live in a fixed 32 MiB array inside the library's own device
 * memory (every GPU that loads the library holds it until the process exits).
 * Calls whose partials need more than that (sinkattn_decode_workspace_bytes)
 * are rejected with SINKATTN_UNSUPPORTED before anything launches. The call
 * allocates nothing and frees nothing.
 *
 * Set-up: the first call in each CUDA context looks up the array's device
 * address (with that context current) and caches it under the context's
 * unique id; make that first call before any stream capture. A new context
 * (after cudaDeviceReset, or a non-primary context made current by another
 * runtime) gets its own lookup on its first call. `stream` must belong to the
 * current device (SINKATTN_INVALID_ARG otherwise, nothing launched): the
 * address is only valid on that device. Every call shares the one array:
 * calls whose kernels may overlap on the GPU (different streams, or several
 * host threads) race on it and must be serialised by the caller. Nothing
 * needs clearing between calls.
 */
SINKATTN_API int sinkattn_decode_noalloc(const void* q, const void* k, const void* v,
                                         const int32_t* kv_indptr, int32_t batch, int32_t q_len,
                                         int32_t max_kv_len, int32_t num_qo_heads,
                                         int32_t num_kv_heads, int32_t head_dim, float sm_scale,
                                         int32_t causal, int32_t window, int32_t num_splits,
                                         const float* sinks, void* out, float* lse, void* stream);

/* Workspace bytes sinkattn_decode needs for these sizes (host only, no CUDA call). */
SINKATTN_API int sinkattn_decode_workspace_bytes(int32_t batch, int32_t q_len, int32_t num_qo_heads,
                                    int32_t head_dim, int32_t num_splits, size_t* bytes);

/*
 * The split count sinkattn_decode and sinkattn_decode_fused use when given
 * num_splits <= 0: enough (sequence, KV head, chunk) work items to fill every
 * SM several times over, without chunks shorter than a few KV tiles; at most
 * 16. Host only; queries the current device's SM count once.
 */
SINKATTN_API int sinkattn_decode_default_splits(int32_t batch, int32_t q_len, int32_t num_qo_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t max_kv_len,
                                   int32_t* num_splits);

/*
 * Which kernel computes the split-KV partials (sinkattn_decode_split, and so
 * sinkattn_decode and sinkattn_decode_noalloc). Process-wide, host only.
 *   SINKATTN_DECODE_AUTO (0, default): the tcgen05 kernel at head_dim 128,
 *     the warp-level kernel at head_dim 64;
 *   SINKATTN_DECODE_WARP (1): the warp-level (mma.sync) kernel;
 *   SINKATTN_DECODE_TCGEN05 (2): the tcgen05/TMEM kernel (head_dim 128;
 *     the query tokens x heads of a GQA group fill up to 128 MMA rows, e.g.
 *     3 MTP tokens x 16 heads = 48); head_dim 64 then returns
 *     SINKATTN_UNSUPPORTED.
 * Both kernels produce the same partial layout and meaning. Returns
 * SINKATTN_INVALID_ARG for any other value.
 */
#define SINKATTN_DECODE_AUTO 0
#define SINKATTN_DECODE_WARP 1
#define SINKATTN_DECODE_TCGEN05 2
SINKATTN_API int sinkattn_set_decode_kernel(int kind);

/*
 * Process-wide choice of the prefill launch (both run the same tcgen05
 * kernel body and give the same results up to floating-point rounding order):
 *   SINKATTN_PREFILL_AUTO (0, default): persistent when the work items are
 *     short (a sliding window, or prompts of a few KV tiles) or when there
 *     are at least 16 items per SM; else one block per item;
 *   SINKATTN_PREFILL_ONE_BLOCK (1): one thread block per (query block, KV
 *     head, sequence), scheduled by the hardware;
 *   SINKATTN_PREFILL_PERSISTENT (2): one thread block per SM working through
 *     a fixed list of items, streaming K/V across item boundaries.
 * Returns SINKATTN_INVALID_ARG for any other value.
 */
#define SINKATTN_PREFILL_AUTO 0
#define SINKATTN_PREFILL_ONE_BLOCK 1
#define SINKATTN_PREFILL_PERSISTENT 2
SINKATTN_API int sinkattn_set_prefill_kernel(int kind);

/*
 * Paged KV cache (HND within a page: heads leading, tokens contiguous): the
 * same operations as sinkattn_prefill, sinkattn_decode_split and
 * sinkattn_decode, with K and V held in page pools
 *   k_pages, v_pages: bf16 [num_pages, Hkv, page_size, d] (device)
 * and sequence b's keys [e * page_size, (e + 1) * page_size) in page
 * page_indices[page_indptr[b] + e]:
 *   page_indptr  int32 [batch + 1] (device), page_indices int32
 *   [page_indptr[batch]] (device), each entry in [0, num_pages).
 * Key counts still come from cu_seqlens_k / kv_indptr (only their
 * differences are used); sequence b needs at least ceil(Lk_b / page_size)
 * pages -- fewer makes the kernel record SINKATTN_BAD_LENGTHS (see
 * sinkattn_debug_status). page_size is a power of two in [16, 256]
 * (SINKATTN_UNSUPPORTED otherwise); num_pages * Hkv * page_size < 2^31.
 * Slots of the last page past Lk_b are read and masked (weight 0): they must
 * hold finite values (a zero-initialised pool does). A page index outside
 * [0, num_pages) gives undefined values for its sequence but no read outside
 * the pools (the copy engine bounds every copy by the pool's extent).
 * Every other argument, layout, rule and result is that of the contiguous
 * entry point; in particular the partials and the merge are the same.
 */
SINKATTN_API int sinkattn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                                        const float* sinks, const int32_t* cu_seqlens_q,
                                        const int32_t* cu_seqlens_k, const int32_t* page_indptr,
                                        const int32_t* page_indices, int32_t num_pages,
                                        int32_t page_size, int32_t batch, int32_t total_q,
                                        int32_t max_seqlen_q, int32_t max_seqlen_k,
                                        int32_t num_qo_heads, int32_t num_kv_heads,
                                        int32_t head_dim, float sm_scale, int32_t causal,
                                        int32_t window, void* out, float* lse, void* stream);
SINKATTN_API int sinkattn_decode_split_paged(const void* q, const void* k_pages,
                                             const void* v_pages, const int32_t* kv_indptr,
                                             const int32_t* page_indptr,
                                             const int32_t* page_indices, int32_t num_pages,
                                             int32_t page_size, int32_t batch, int32_t q_len,
                                             int32_t max_kv_len, int32_t num_qo_heads,
                                             int32_t num_kv_heads, int32_t head_dim,
                                             float sm_scale, int32_t causal, int32_t window,
                                             int32_t num_splits, float* part_acc, float* part_md,
                                             void* stream);
SINKATTN_API int sinkattn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* kv_indptr, const int32_t* page_indptr,
                                       const int32_t* page_indices, int32_t num_pages,
                                       int32_t page_size, int32_t batch, int32_t q_len,
                                       int32_t max_kv_len, int32_t num_qo_heads,
                                       int32_t num_kv_heads, int32_t head_dim, float sm_scale,
                                       int32_t causal, int32_t window, int32_t num_splits,
                                       const float* sinks, void* workspace,
                                       size_t workspace_bytes, void* out, float* lse,
                                       void* stream);

/*
 * FP8 KV cache: sinkattn_decode_split and sinkattn_decode with K and V held
 * as e4m3 codes (the OCP 8-bit floating-point format E4M3, one byte per
 * element, in the same ragged HND layout) and per-KV-head fp32 scales:
 *   k, v:     uint8 codes [Hkv * total_k, d] (device);
 *   k_scale:  float [Hkv] (device): key j of KV head g is code * k_scale[g];
 *   v_scale:  float [Hkv] (device): value j of KV head g is code * v_scale[g].
 * Every other argument, layout, result, the partials and the merge are those
 * of the bf16 entry points ("GPT-OSS on Day 0", section "Kernels for GPT-OSS /
 * Sink attention", with the keys and values dequantised). The kernel widens
 * the codes to f16, which holds every e4m3 value exactly, and runs the
 * products in f16 with q converted to f16: |q| must stay below 65504, and
 * q elements below 2^-14 in magnitude lose relative precision. Kernel
 * choice (sinkattn_set_decode_kernel): at head_dim 128 with at most 64 query
 * heads per KV head the tcgen05 kernel runs (AUTO or TCGEN05), other shapes
 * take the warp-level kernel (TCGEN05 forced there: SINKATTN_UNSUPPORTED).
 * k_scale / v_scale null or misaligned: SINKATTN_INVALID_ARG.
 */
SINKATTN_API int sinkattn_decode_split_fp8(const void* q, const void* k, const void* v,
                                           const float* k_scale, const float* v_scale,
                                           const int32_t* kv_indptr, int32_t batch,
                                           int32_t q_len, int32_t max_kv_len,
                                           int32_t num_qo_heads, int32_t num_kv_heads,
                                           int32_t head_dim, float sm_scale, int32_t causal,
                                           int32_t window, int32_t num_splits, float* part_acc,
                                           float* part_md, void* stream);
SINKATTN_API int sinkattn_decode_fp8(const void* q, const void* k, const void* v,
                                     const float* k_scale, const float* v_scale,
                                     const int32_t* kv_indptr, int32_t batch, int32_t q_len,
                                     int32_t max_kv_len, int32_t num_qo_heads,
                                     int32_t num_kv_heads, int32_t head_dim, float sm_scale,
                                     int32_t causal, int32_t window, int32_t num_splits,
                                     const float* sinks, void* workspace,
                                     size_t workspace_bytes, void* out, float* lse,
                                     void* stream);

/* Human-readable name of a status code (static string). */
SINKATTN_API const char* sinkattn_status_string(int status);

/* Description of the last error returned on this thread ("" if none). */
SINKATTN_API const char* sinkattn_last_error(void);

/*
 * Diagnostic, not for the hot path: synchronises `stream`, then reads and
 * clears the device status word of every kernel in the library. *status gets
 * SINKATTN_OK, SINKATTN_TIMEOUT or SINKATTN_BAD_LENGTHS. Returns
 * SINKATTN_CUDA_ERROR if the synchronisation or the read failed.
 */
SINKATTN_API int sinkattn_debug_status(void* stream, int* status);

/*
 * Diagnostic, test only (failure detection without a GPU fault; the pages
 * have no counterpart): sets, for every kernel of the library, the number of
 * SM clock cycles a bounded wait allows before it gives up
 * (wait_limit_cycles <= 0 restores the default, about 1 s), and makes the
 * TMA producer of the first thread block of every later launch leave out the
 * copies of its KV tile number skip_tile (-1: none). A left-out tile's
 * waits run out: the kernel records SINKATTN_TIMEOUT (read by
 * sinkattn_debug_status), drains its copies and MMAs, frees its tensor
 * memory and exits; its outputs are then undefined. Host call, synchronous
 * with the device; make it while no kernel of the library is running.
 * skip_tile < -1: SINKATTN_INVALID_ARG.
 */
SINKATTN_API int sinkattn_debug_set_hooks(long long wait_limit_cycles, int skip_tile);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H_ */
