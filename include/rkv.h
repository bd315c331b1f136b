/*
 * rkv.h -- C ABI of librkv, a GB300 (sm_103a) implementation of RocketKV's
 * decode-time hot path: stage-1 SnapKV++ eviction at prefill and stage-2 Hybrid
 * Sparse Attention (HSA) at every decode step.
 *
 * Sources, cited by short name:
 *   [summary]  "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage
 *              KV Cache Compression", research-map summary, sections Problem,
 *              Approach, Key results.
 *   [abstract] the same paper's abstract (arXiv 2502.14051).
 *   [adapted]  "RocketKV-adapted -- Two-Stage Compression (SnapKV Eviction +
 *              Hybrid Sparse Attention)", VeloxQuant-MLX docs, sections "Where
 *              it sits -- the mechanism gap", "The one setting worth tuning:
 *              rocketkv_compression_ratio", "Adaptation notes", "Evidence".
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers, 16-byte aligned, owned by
 *     the caller.  The library never allocates or frees device memory and keeps no
 *     per-cache state; scratch lives in a caller-provided workspace.
 *   - Pointers marked "host" are read during the call only.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and returns without synchronising, except rkv_get_device_status.
 *   - Arguments are validated on the host before anything is enqueued; a failed
 *     check returns RKV_ERR_INVALID_ARG / RKV_ERR_UNSUPPORTED / RKV_ERR_WORKSPACE
 *     with no side effect and a message in rkv_last_error().
 *   - A failed kernel launch returns RKV_ERR_CUDA.
 *   - Errors found on the device (a page id out of range, a sequence longer than
 *     its pages, a bounded wait that ran out) are OR-ed into cache->error_word as
 *     RKV_DEVERR_* bits; the kernel skips the offending access and carries on.
 *     rkv_get_device_status reads and clears the word.
 *   - head_dim must be 128; page_size 16, 32 or 64; Hq a multiple of Hkv with
 *     G = Hq / Hkv in {1, 2, 4, 8}.
 *   - bf16 data is passed as IEEE bfloat16 bit patterns (rkv_bf16).
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t rkv_bf16;

typedef enum {
  RKV_OK = 0,
  RKV_ERR_INVALID_ARG = 1,
  RKV_ERR_UNSUPPORTED = 2,
  RKV_ERR_WORKSPACE = 3,
  RKV_ERR_CUDA = 4,
  RKV_ERR_DEVICE_DATA = 5,
  RKV_ERR_TIMEOUT = 6
} rkv_status;

/* bits of cache->error_word */
#define RKV_DEVERR_PAGE_ID   0x1  /* page_table entry outside [0, num_phys_pages) */
#define RKV_DEVERR_CAPACITY  0x2  /* seq_len (+ appended tokens) beyond max_pages * page_size */
#define RKV_DEVERR_TIMEOUT   0x4  /* a bounded wait on an mbarrier ran out */
#define RKV_DEVERR_SEQ_LEN   0x8  /* device seq_len differs from the held_len the host passed */

#define RKV_HEAD_DIM 128
#define RKV_MAX_BATCH 256

/* Result of the adaptive ratio split. */
typedef struct {
  double c;          /* overall ratio prompt_len / budget */
  double r;          /* stage-1 share of log c */
  double c1;         /* stage-1 (eviction) ratio c^r */
  double c2;         /* stage-2 (HSA) ratio c^(1-r) */
  int32_t keep1;     /* stage-1 survivors per KV head, window included */
  int32_t k1;        /* HSA channels per KV head */
  int32_t k2;        /* HSA pages per KV head per step */
  int32_t pool_kernel; /* default stage-1 max-pool kernel for this prompt length */
} rkv_split;

/*
 * The compressed, paged KV cache of one attention layer (all device memory,
 * caller-owned).
 *   k_pages, v_pages : [num_phys_pages][Hkv][page_size][head_dim] bf16.  Token i of
 *                      sequence b sits in physical page page_table[b][i / page_size],
 *                      slot i % page_size.  Survivors are stored in ascending
 *                      original position, decode tokens after them.
 *   page_table       : [B][max_pages] int32 physical page ids.
 *   seq_len          : [B] int32, current compressed length n of each sequence.
 *   kmax, kmin       : [B][Hkv][head_dim][max_pages] bf16, channel-major paged
 *                      element-wise max / min of the keys ([adapted], "Where it
 *                      sits": Quest-style paged max/min summaries).  Only pages
 *                      below ceil(n / page_size) are meaningful.
 *   error_word       : one device int32 receiving RKV_DEVERR_* bits.
 *   step_sync        : [B] int32, zero when the cache is created; rkv_decode_step
 *                      uses it to advance seq_len exactly once per sequence and
 *                      leaves it at zero.  May be NULL if rkv_decode_step is not used.
 * max_pages must be a multiple of 8 and at most 16384, and num_phys_pages * Hkv *
 * page_size below 2^31 (RKV_ERR_UNSUPPORTED otherwise).
 */
typedef struct {
  rkv_bf16* k_pages;
  rkv_bf16* v_pages;
  int32_t* page_table;
  int32_t* seq_len;
  rkv_bf16* kmax;
  rkv_bf16* kmin;
  int32_t* error_word;
  int32_t* step_sync;
  int32_t B, Hkv, head_dim, page_size, max_pages, num_phys_pages;
} rkv_cache;

/*
 * Adaptive split of the overall ratio c = prompt_len / budget between the stages
 * ([adapted], "The one setting worth tuning"): r = clip(0.2 + 0.06*log2(c), 0.2,
 * 0.8), stage 1 compresses by c^r and stage 2 by c^(1-r) (c = 64 -> 10.3x / 6.2x).
 * Sizes (readings; the pages leave them open): keep1 = round(prompt_len / c^r)
 * clamped to [max(budget, window), prompt_len]; k2 = budget / page_size;
 * k1 = 16*round(head_dim / (16*sqrt(c2))) in [16, head_dim] unless k1_override > 0;
 * pool_kernel = 7 / 31 / 63 for prompts up to 8K / 48K / longer.
 * Host only.  Returns RKV_ERR_INVALID_ARG for non-positive sizes or out == NULL.
 */
rkv_status rkv_split_ratio(int32_t prompt_len, int32_t budget, int32_t head_dim,
                           int32_t page_size, int32_t window, int32_t k1_override,
                           rkv_split* out);

/*
 * The split of RocketKV-MT ("RocketKV: Accelerating Long-Context LLM Inference via
 * Two-Stage KV Cache Compression", research-map summary, "Approach": the variant
 * that retains the tokens stage 1 would evict; "RocketKV-adapted", "Should you use
 * this?": it skips permanent eviction).  Nothing is evicted (keep1 = prompt_len,
 * c1 = 1, r = 0) and HSA takes the whole ratio c = prompt_len / budget as c2; k1,
 * k2 and pool_kernel follow the same rules as rkv_split_ratio with that c2.  Passing
 * this keep1 to rkv_prefill_evict builds the paged cache and summaries over the whole
 * prompt and skips the stage-1 scoring.  Host only.
 */
rkv_status rkv_split_ratio_mt(int32_t prompt_len, int32_t budget, int32_t head_dim,
                              int32_t page_size, int32_t k1_override, rkv_split* out);

/* Bytes of workspace rkv_prefill_evict needs for these sizes. */
size_t rkv_prefill_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t window,
                                  int32_t max_prompt_len);

/*
 * Stage 1, SnapKV++ eviction ([abstract]; [summary], Approach: SnapKV with a
 * large pooling kernel and GQA-group-level selection).  Per sequence b and KV
 * head g:
 *   S[t]  = sum over the G query heads of group g and the w window rows j of
 *           softmax(q_win . k^T * scale)[j, t], row j (prompt position L-w+j)
 *           normalised over the keys t <= L-w+j; scored for t < L-w;
 *   S'    = centred max-pool of S with kernel pool_kernel[b] (out-of-range
 *           positions ignored);
 *   kept  = the top keep1[b]-w positions by (S' desc, position asc) plus the w
 *           window positions, ascending;
 * then the kept tokens' K and V are written into the cache pages (positions
 * 0..keep1-1), their Kmax/Kmin summaries are built and seq_len[b] = keep1[b].
 *   q_win  : device [B][Hq][window][128] bf16, the last `window` queries.
 *   k, v   : device [B][Hkv][max_prompt_len][128] bf16; rows >= prompt_len[b]
 *            are never read.  v may instead be pinned host memory (cudaHostAlloc or
 *            registered, mapped into the device's address space; 16-byte aligned):
 *            only the kept rows of V are read, once, through the mapping, so a
 *            prompt that lives on the host needs only q_win and k copied to the
 *            device (the kernels read nothing else of v).
 *   prompt_len, keep1, pool_kernel : host [B]; window <= keep1[b] <= prompt_len[b]
 *            <= max_prompt_len; pool_kernel odd in [1, 255]; G * window <= 128.
 *   scale  : softmax scale (1/sqrt(128) for the standard one).
 *   cache  : destination; its pages must hold keep1[b] tokens of every sequence.
 *   kept_idx : device [B][Hkv][kept_stride] int32, receives the kept positions.
 *   pooled_scores : device [B][Hkv][max_prompt_len] fp32 receiving S' for
 *            t < L-w, or NULL.
 * When no sequence evicts anything (keep1[b] == prompt_len[b] for every b, as
 * rkv_split_ratio_mt gives) the stage-1 scoring is skipped: kept_idx receives every
 * position and pooled_scores is left untouched.
 */
rkv_status rkv_prefill_evict(const rkv_bf16* q_win, const rkv_bf16* k, const rkv_bf16* v,
                             int32_t B, int32_t Hq, int32_t window, int32_t max_prompt_len,
                             const int32_t* prompt_len, const int32_t* keep1,
                             const int32_t* pool_kernel, float scale,
                             const rkv_cache* cache, int32_t* kept_idx, int32_t kept_stride,
                             float* pooled_scores, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Bytes of workspace rkv_prefill_chunk needs when held_len[b] + chunk_len[b] <= max_total_len. */
size_t rkv_prefill_chunk_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t window,
                                        int32_t max_total_len);

/*
 * Stage 1 over a prompt that arrives in chunks, the budget re-enforced at every
 * chunk ([adapted], "Evidence": stage-1 eviction holds its budget across
 * chunked-prefill calls).  Reading taken: the chunk's tokens join the n_b =
 * held_len[b] + chunk_len[b] tokens held so far (the cache's tokens first, in
 * cache order), and SnapKV++ as in rkv_prefill_evict runs over that sequence with
 * prompt_len = n_b and keep1 = min(keep1[b], n_b), the chunk's last `window` queries
 * being the observation window.  The survivors are written back to the cache's
 * pages from position 0, their summaries rebuilt, seq_len[b] = min(keep1[b], n_b).
 * A sequence with n_b <= keep1[b] keeps everything; when that holds for every b the
 * scoring is skipped.  Start from an empty cache (seq_len 0) for the first chunk.
 *   q_win    : device [B][Hq][window][128] bf16, the chunk's last `window` queries.
 *   k_chunk, v_chunk : device [B][Hkv][chunk_max][128] bf16; rows >= chunk_len[b]
 *              are never read.
 *   chunk_len, held_len, keep1, pool_kernel : host [B]; window <= chunk_len[b] <=
 *              chunk_max; held_len[b] must equal the cache's seq_len[b] (the device
 *              checks it: a mismatch sets RKV_DEVERR_SEQ_LEN); keep1[b] >= window.
 *   cache    : read (the held tokens) and rewritten in place; the held tokens are
 *              copied to the workspace before any page is written.
 *   kept_idx : device [B][Hkv][kept_stride] int32, receives the kept positions of
 *              the n_b-token sequence, ascending.
 *   workspace: rkv_prefill_chunk_workspace_size(B, Hq, Hkv, window, max_b n_b)
 *              bytes or more.
 */
rkv_status rkv_prefill_chunk(const rkv_bf16* q_win, const rkv_bf16* k_chunk, const rkv_bf16* v_chunk,
                             int32_t B, int32_t Hq, int32_t window, int32_t chunk_max,
                             const int32_t* chunk_len, const int32_t* held_len,
                             const int32_t* keep1, const int32_t* pool_kernel, float scale,
                             const rkv_cache* cache, int32_t* kept_idx, int32_t kept_stride,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Append n_new tokens to every sequence and bring the page summaries up to date
 * ([adapted], "Evidence": the incremental update equals a rebuild, bit for bit).
 * For each b the tokens go to positions [seq_len[b], seq_len[b] + n_new): when
 * k_new is not NULL they are first copied from k_new / v_new (device
 * [B][Hkv][n_new][128] bf16) into their page slots, otherwise they must already
 * be there.  Every touched page's Kmax/Kmin is brought up to date: with k_new, a
 * page's stored summary (of its earlier tokens) is folded with the new keys; without,
 * the page is recomputed from its valid tokens.  Then seq_len[b] += n_new.  With seq_len = 0 and n_new = n this is a full
 * rebuild.  A sequence that would outgrow its pages is left unchanged and flags
 * RKV_DEVERR_CAPACITY.
 */
rkv_status rkv_append_page_summary(const rkv_cache* cache, const rkv_bf16* k_new,
                                   const rkv_bf16* v_new, int32_t n_new, void* stream);

/* Bytes of workspace rkv_decode_hsa and rkv_decode_step need. */
size_t rkv_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_pages);

/*
 * Stage 2, one Hybrid Sparse Attention step over the current cache ([adapted],
 * "Where it sits" and "Adaptation notes"; [abstract]).  Per sequence b and KV
 * head g, with n = seq_len[b] and NP = ceil(n / page_size):
 *   1. channels S = top-k1[b] of a_i = sum over the group's heads of |q_h,i|
 *      (ties: lower channel);
 *   2. page bound s_p = sum_h sum_{i in S} max(q_h,i*Kmax_i,p, q_h,i*Kmin_i,p);
 *   3. pages = top-min(k2[b], NP) by (s_p desc, page asc);
 *   4. out_h = softmax(q_h . k_t * scale) . v_t over all 128 channels of every
 *      valid token t < n of the selected pages, for each head h of the group.
 *   q            : device [B][Hq][128] bf16 decode queries.
 *   k1, k2       : host [B]; 1 <= k1 <= 128, k2 >= 1.
 *   out          : device [B][Hq][128] fp32.
 *   sel_channels : device [B][Hkv][128] int32 or NULL; receives the channel set,
 *                  ascending, in the first k1[b] entries.
 *   sel_pages    : device [B][Hkv][sel_pages_stride] int32 or NULL; receives the
 *                  page set, ascending, in the first min(k2[b], NP) entries and -1
 *                  in the next entry if there is room.
 */
rkv_status rkv_decode_hsa(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq,
                          const int32_t* k1, const int32_t* k2, float scale, float* out,
                          int32_t* sel_channels, int32_t* sel_pages, int32_t sel_pages_stride,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * One whole decode step: append one token to every sequence, then the HSA step of
 * rkv_decode_hsa over the grown cache (the new token is a candidate like any
 * other).  Equivalent to rkv_append_page_summary(cache, k_new, v_new, 1) followed
 * by rkv_decode_hsa, but while max_pages <= 4096 it runs as one kernel launch:
 * one thread-block cluster per (sequence, KV head) shares its page scores and its
 * partial softmax states through distributed shared memory.
 *   k_new, v_new : device [B][Hkv][128] bf16, the new token's key and value.
 *   cache->step_sync must be set (zero-initialised with the cache).
 * Other arguments as for rkv_decode_hsa; the workspace is used only by the
 * multi-kernel path for larger caches.
 */
rkv_status rkv_decode_step(const rkv_cache* cache, const rkv_bf16* q, const rkv_bf16* k_new,
                           const rkv_bf16* v_new, int32_t Hq, const int32_t* k1, const int32_t* k2,
                           float scale, float* out, int32_t* sel_channels, int32_t* sel_pages,
                           int32_t sel_pages_stride, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Bytes of device staging rkv_decode_step_host needs: the packed inputs, then out. */
size_t rkv_step_host_staging_size(int32_t B, int32_t Hq, int32_t Hkv);

/*
 * rkv_decode_step with the step's inputs and output in host memory, for a caller
 * whose tensors live on the host (pinned memory keeps the copies asynchronous).
 *   host_in  : host, packed bf16: q [B][Hq][128], then k_new [B][Hkv][128], then
 *              v_new [B][Hkv][128], contiguous.
 *   host_out : host [B][Hq][128] fp32, written when the stream reaches the copy back.
 *   staging  : device, rkv_step_host_staging_size(B, Hq, Hkv) bytes or more, 16-byte
 *              aligned; receives the inputs (one host-to-device copy) and out.
 * When both host buffers are pinned memory mapped into the device's address space
 * (cudaHostAlloc / torch pin_memory, with unified addressing) and 16-byte aligned, the
 * step's kernel reads the inputs and writes out through that mapping and nothing is
 * copied; otherwise it enqueues on `stream` the input copy, the decode step and the
 * output copy (one device-to-host copy).  Other arguments as for rkv_decode_step.
 */
rkv_status rkv_decode_step_host(const rkv_cache* cache, const void* host_in, float* host_out,
                                int32_t Hq, const int32_t* k1, const int32_t* k2, float scale,
                                void* staging, size_t staging_bytes, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Which implementation rkv_decode_hsa / rkv_decode_step use, process-wide:
 * 0 = automatic (the fused one-launch kernel whenever max_pages <= 4096),
 * 1 = always the four-kernel path, 2 = fused when possible (as 0).  Any other
 * value leaves the setting unchanged.  Returns the setting in force.  Both paths
 * compute the same result; this exists for testing and measurement.
 */
int32_t rkv_decode_path(int32_t path);

/*
 * rkv_decode_hsa without a workspace argument, for callers that cannot allocate
 * device memory when they call (for instance a plug-in inside an engine that owns
 * every device allocation, or a latency-critical loop that must never reach
 * cudaMalloc and its device-wide synchronisation).  The pages describe no such
 * call; it exists for those callers only.  It computes exactly what
 * rkv_decode_hsa computes, using as scratch one array of 32 MiB compiled into the
 * library (held on every GPU that loads the library until the process exits).
 *   - It allocates nothing and frees nothing.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call outside any stream
 *     capture.
 *   - A cache whose rkv_decode_workspace_size exceeds 32 MiB is rejected with
 *     RKV_ERR_WORKSPACE and nothing is launched.
 *   - All calls share the one array: two calls whose work overlaps on the GPU (on
 *     different streams, or from different threads) race and corrupt each other;
 *     order them on one stream.  Nothing in the array needs to start at zero.
 * Arguments, layouts and other statuses as for rkv_decode_hsa.
 */
rkv_status rkv_decode_hsa_noalloc(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq,
                                  const int32_t* k1, const int32_t* k2, float scale, float* out,
                                  int32_t* sel_channels, int32_t* sel_pages,
                                  int32_t sel_pages_stride, void* stream);

/* Bytes of workspace rkv_decode_sparq needs. */
size_t rkv_sparq_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_pages,
                                int32_t page_size);

/*
 * SparQ-only selection: HSA with one-token pages (RocketKV summary, ablation of the
 * two halves of HSA: SparQ's channel selection alone; "RocketKV-adapted", "Where it
 * sits -- the mechanism gap": SparQ-style top-magnitude channels along the head
 * dimension).  Reading taken: with a page of one token, Kmax = Kmin = the key, so the
 * page bound of rkv_decode_hsa becomes the key's partial dot product over the chosen
 * channels.  Per sequence b and KV head g, with n = seq_len[b]:
 *   1. channels S = top-k1[b] of sum over the group's heads of |q_h,i| (ties: lower);
 *   2. s_t = sum_h sum_{i in S} q_h,i k_t,i for every cached token t < n, read from
 *      the cache's key rows (any page_size);
 *   3. tokens = top-min(k_tokens[b], n) by (s_t desc, t asc);
 *   4. out_h = softmax(q_h . k_t * scale) . v_t over all 128 channels of those tokens.
 * Arguments as rkv_decode_hsa, with k_tokens (host [B], >= 1) in place of k2 and
 * sel_tokens (device [B][Hkv][sel_tokens_stride] int32, ascending, then -1 when there
 * is room; may be NULL) in place of sel_pages.  No append: call
 * rkv_append_page_summary first.  Caches of more than 32768 tokens per sequence
 * (max_pages * page_size) return RKV_ERR_UNSUPPORTED.
 * keys_t (may be NULL): a channel-major copy of the cached keys, the layout SparQ
 * scores from (each chosen channel's values of every position contiguous, so step 2
 * reads k1 of the 128 channels): device, 16-byte aligned, keys_t_bytes >=
 * rkv_sparq_keys_size(B, Hkv, max_pages, page_size) (else RKV_ERR_WORKSPACE).  It is
 * owned by the caller and kept between calls: it starts zero-filled (empty), and each
 * call first copies into it the positions the cache gained since the previous call
 * (all of them the first time), then scores from it.  Zero it again whenever the
 * cache's positions are rewritten rather than appended (a new prefill).  The
 * selections and the output are those of the call without it, up to the fp32 order
 * of the partial dot products.  With NULL, step 2 reads the cache's key rows.
 */
rkv_status rkv_decode_sparq(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq,
                            const int32_t* k1, const int32_t* k_tokens, float scale, float* out,
                            int32_t* sel_channels, int32_t* sel_tokens, int32_t sel_tokens_stride,
                            void* keys_t, size_t keys_t_bytes, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Bytes of the channel-major key copy rkv_decode_sparq can keep and score from:
 * a [B*Hkv] int32 record of the positions copied (256-byte padded), then per (b, g)
 * a [128][max_pages * page_size] bf16 block. */
size_t rkv_sparq_keys_size(int32_t B, int32_t Hkv, int32_t max_pages, int32_t page_size);

/*
 * Exact-TopK recall of a page selection: a diagnostic, not a step of the method.
 * The summary page of "RocketKV: Accelerating Long-Context LLM Inference via
 * Two-Stage KV Cache Compression" measures RocketKV against the Exact-TopK
 * baseline ("Surprising findings", "Limitations"); "RocketKV-adapted" compares
 * selections by overlap with an oracle top-k ("Where it sits -- the mechanism gap",
 * "Evidence").
 * For every (sequence b, KV head g) of the cache as it stands (n = seq_len[b]
 * tokens), with the group's query heads q[b][g*G .. g*G+G):
 *   e_t = sum over the group's heads h of softmax over t < n of (q_h . k_t * scale)
 *   top = the K = min(k_tokens[b], n) tokens of largest e_t (ties: lower index)
 *   recall[b*Hkv+g] = |top tokens inside the selected pages| / K      (1 when K = 0)
 *   mass[b*Hkv+g]   = (e_t summed over those) / (e_t summed over top)  (may be NULL)
 * sel_pages: device [B][Hkv][sel_pages_stride] page ids as rkv_decode_hsa writes
 * them (ascending; a -1 ends a shorter list; ids outside [0, NP) are ignored).
 * k_tokens: HOST [B] (the stage-2 token budget, k2 * page_size).  q: device
 * [B][Hq][128] bf16; recall, mass: device [B*Hkv] fp32; 16-byte aligned.
 * Supports n <= 49152 per sequence (RKV_ERR_UNSUPPORTED if the cache could hold
 * more).  Reads every cached key twice.  Bad page ids set RKV_DEVERR_PAGE_ID.
 */
rkv_status rkv_exact_topk_recall(const rkv_cache* cache, const rkv_bf16* q, int32_t Hq,
                                 const int32_t* sel_pages, int32_t sel_pages_stride,
                                 const int32_t* k_tokens, float scale, float* recall, float* mass,
                                 void* stream);

/*
 * Self-test of the device failure path (not a step of the method; the pages describe
 * no GPU code).  Every wait of the library's kernels on an mbarrier (a TMA or bulk
 * copy landing, another warp's hand-off) gives up after 1 s, sets RKV_DEVERR_TIMEOUT
 * in cache->error_word, drains what it issued and returns, so a stall never hangs the
 * GPU.  This call launches one CTA that waits, for at most limit_ns nanoseconds
 * (1 <= limit_ns <= 1e9), on an mbarrier nothing arrives on and no copy targets; the
 * wait runs out and the bit is set exactly as a stalled kernel would set it, so that
 * rkv_get_device_status then returns RKV_ERR_TIMEOUT.  Only error_word is touched.
 */
rkv_status rkv_selftest_bounded_wait(const rkv_cache* cache, int64_t limit_ns, void* stream);

/* Synchronise `stream`, read and clear cache->error_word.  RKV_OK when it was 0,
 * RKV_ERR_TIMEOUT when the timeout bit was set, else RKV_ERR_DEVICE_DATA; *bits
 * (if not NULL) receives the raw word. */
rkv_status rkv_get_device_status(const rkv_cache* cache, void* stream, int32_t* bits);

/* Message of the last failed call on this thread ("" if none). */
const char* rkv_last_error(void);

/* Number of kernels this library has launched in this process. */
int64_t rkv_launch_count(void);

/*
 * Per-kernel timing for measurement.  While enabled, every kernel launch is
 * bracketed by a pair of CUDA events recorded on its own stream (inside a stream
 * capture the records become graph nodes, re-recorded on every replay).
 * rkv_profile_accumulate synchronises every recorded pair and adds its elapsed
 * time to per-kind totals, keeping the pairs (call it after each graph replay);
 * rkv_profile_release frees the pairs; rkv_profile_reset zeroes the totals;
 * rkv_profile_read returns a kind's launch count and summed device time (ms) and
 * its name, or NULL past the last kind.  Host only; not for use in hot loops.
 */
void rkv_profile_enable(int32_t enable);
void rkv_profile_accumulate(void);
void rkv_profile_release(void);
void rkv_profile_reset(void);
const char* rkv_profile_read(int32_t kind, int64_t* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* RKV_H */
