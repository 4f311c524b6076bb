/*
 * sls.h - C ABI of the GB300 sparse decode-attention library (libsls.so).
 *
 * One decode step of sparse long-context attention:
 *
 *   select   sls_select_pages   Quest-style page bound + per-KV-head top-k
 *            sls_select_delta   2-bit thumbnail scan + top-delta
 *   attend   sls_sparse_decode_attend   split-K online softmax over the
 *                                       selected pages (flash-decoding)
 *   combine  sls_combine_splits         log-sum-exp merge of the splits,
 *                                       with the optional sink
 *
 * plus the selector metadata kept next to the KV cache (page min/max keys,
 * 2-bit thumbnails), built in bulk or updated on append.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *   stated otherwise.  The library allocates no memory; scratch comes from a
 *   caller buffer whose size a *_workspace_size() call reports.
 * - Queries, K/V caches, page metadata (kmin/kmax), thumbnail codes, scales
 *   and residuals, appended keys/values and split partials (o_part) are read
 *   in 16-byte vectors: their pointers must be 16-byte aligned, or the call
 *   fails with SLS_EINVAL before launching anything.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Calls only enqueue work: they never synchronise the device
 *   and never read device memory from the host, so they can be captured in
 *   a CUDA graph.
 * - Every call returns an sls_status.  Arguments are validated on the host
 *   before anything is launched; on error nothing is enqueued and
 *   sls_last_error() describes the problem (thread-local string).
 * - KV cache layout: K and V are [B, Hkv, Cap, D] row-major, element type
 *   desc->dtype.  Row r = b*Hkv + h of the cache is the contiguous slice of
 *   request (b, kv head h); seen as a page pool it holds Cap/P pages of P
 *   tokens, page p covering positions [p*P, p*P+P) ("perf(core): fused
 *   sparse-attention decode via page indirection", section "The reduction":
 *   a dense [B, H, Cap, D] allocation viewed as a pool by a pure reshape,
 *   with the KV-head axis folded into the request axis).
 * - Query heads: q is [B, Hq, D]; query head hq belongs to KV head
 *   hq / (Hq/Hkv) (grouped-query attention), and every page list is shared
 *   by the G = Hq/Hkv query heads of its KV head.
 * - ctx_len[b] is the number of valid positions of sequence b; positions
 *   >= ctx_len[b] are never read by selection and never attended.  Values
 *   outside [0, Cap] are clamped to that range on the device.
 * - Page indices in page lists are LOGICAL page numbers within the row
 *   (0 .. Cap/P - 1); -1 marks an empty slot that is skipped.
 */
#ifndef SLS_H
#define SLS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
typedef int sls_status;
#define SLS_OK            0
#define SLS_EINVAL       -1  /* null pointer, bad size or out-of-range parameter */
#define SLS_EUNSUPPORTED -2  /* valid but unsupported combination (dtype, D, G, P) */
#define SLS_EOVERFLOW    -3  /* a size product overflows the index range */
#define SLS_EWORKSPACE   -4  /* workspace missing or too small */
#define SLS_ECUDA        -5  /* a CUDA launch or attribute call failed */
#define SLS_ETIMEOUT     -6  /* a pipelined kernel gave up waiting for its own copies */
#define SLS_EDEVICE      -7  /* a kernel met page-list entries it could not use (skipped) */

/* ---- element types ----------------------------------------------------- */
#define SLS_DTYPE_F32  0
#define SLS_DTYPE_BF16 1

/* ---- descriptor flags -------------------------------------------------- */
/* Use the CUDA-core kernels even where a tensor-core kernel exists (for
 * comparison; results agree within the same tolerances). */
#define SLS_FLAG_CUDA_CORES 1
/* Feed the bf16 tensor-core attend kernel from registers (16-byte loads)
 * instead of the shared-memory ring filled by tensor-map copies (for
 * comparison; results agree within the same tolerances). */
#define SLS_FLAG_NO_TMA 2
/* Test hook of the bounded waits, not for production: in the tensor-map fed
 * kernels (sls_sparse_decode_attend[_combine] on bf16 pages of >= 16 tokens,
 * and the one-launch sls_quest_decode_step), the first CTA of the launch
 * announces 16 bytes on its first attend stage that it never requests, and
 * that CTA's waits poll a short while only.  The waits on that stage
 * give up, the first row's outputs become NaN, and the next
 * sls_pipeline_check() returns SLS_ETIMEOUT.  No copy is issued for the
 * announced bytes, so nothing faults and nothing waits forever. */
#define SLS_FLAG_TEST_WAIT_TIMEOUT 4

/*
 * Shapes and element type of one attention layer's decode step.
 *   batch        B >= 1
 *   num_q_heads  Hq >= 1
 *   num_kv_heads Hkv >= 1, Hq % Hkv == 0, G = Hq/Hkv <= 8
 *   head_dim     D in {64, 128}
 *   page_size    P, a power of two in [1, 256]; Cap % P == 0
 *   capacity     Cap >= 1 cache slots per (b, kv head)
 *   dtype        SLS_DTYPE_F32 or SLS_DTYPE_BF16: K, V, q, page min/max,
 *                thumbnail scales and the combined output use this type
 *   flags        bitwise OR of SLS_FLAG_* (0 by default)
 *   scale        softmax scale applied to q.k; 0 selects 1/sqrt(D)
 *                ("Attention: Undivided & Uncompressed", Notation:
 *                S = QK^T / sqrt(d))
 */
typedef struct sls_attn_desc {
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t capacity;
  int32_t dtype;
  int32_t flags;
  float scale;
} sls_attn_desc;

/* ---- metadata: Quest page min/max -------------------------------------- */

/*
 * Per-page, per-channel min and max of the keys ("Don't read the haystack",
 * Part two: for each page keep the elementwise min and max of its keys).
 *   k_cache  [B, Hkv, Cap, D]  dtype            (read)
 *   ctx_len  [B] int32                          (read)
 *   kmin     [B, Hkv, Cap/P, D] dtype           (written)
 *   kmax     [B, Hkv, Cap/P, D] dtype           (written)
 * Pages p < ceil(ctx_len[b]/P) are written; a partial last page summarises
 * only its positions < ctx_len[b]; later pages are left untouched.  The
 * stored values are exact copies of key elements.
 */
sls_status sls_pagemeta_build(const sls_attn_desc* desc, const void* k_cache,
                              const int32_t* ctx_len, void* kmin, void* kmax,
                              void* stream);

/*
 * Fold one appended key per sequence into its page's min/max ("Don't read
 * the haystack", Part two: summaries maintained incrementally as tokens
 * append).  The caller has already written the key at position pos[b] of
 * every kv head of sequence b.  When pos[b] % P == 0 the page is reset to
 * that key; otherwise min/max are taken with the stored values.  pos[b] < 0
 * skips sequence b; pos[b] >= Cap is clamped away (skipped) on the device.
 *   k_cache [B, Hkv, Cap, D] (read), pos [B] int32 (read),
 *   kmin, kmax [B, Hkv, Cap/P, D] (read-modify-write)
 */
sls_status sls_pagemeta_update(const sls_attn_desc* desc, const void* k_cache,
                               const int32_t* pos, void* kmin, void* kmax,
                               void* stream);

/*
 * Append one decoded token per sequence, entirely on the device, so that a
 * captured decode step can be replayed step after step: the new key and
 * value of every KV head are written at position ctx_len[b], the key is
 * folded into its page's min/max as sls_pagemeta_update does ("Don't read
 * the haystack", Part two: summaries maintained as tokens append), and
 * ctx_len[b] advances by one.  A sequence already at capacity is left
 * unchanged.
 *   k_new, v_new  [B, Hkv, D] dtype (read)
 *   k_cache, v_cache  [B, Hkv, Cap, D] dtype (row ctx_len[b] written)
 *   kmin, kmax    page metadata to keep current, or both NULL (page size 1,
 *                 or a selector without it)
 *   ctx_len       [B] int32 (read and advanced)
 *   pos_out       [B] int32 receiving the written position (-1 at capacity),
 *                 e.g. for sls_thumb_update; may be NULL
 */
sls_status sls_decode_append(const sls_attn_desc* desc, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, void* kmin, void* kmax,
                             int32_t* ctx_len, int32_t* pos_out, void* stream);

/* ---- metadata: 2-bit key thumbnails ------------------------------------ */

/*
 * 2-bit symmetric zero-free (mid-rise) thumbnails of every complete block
 * of `block` tokens ("Faster Than Flash", Methodology 1): per block and
 * channel s = max|k|; each key element gets a 2-bit code for the levels
 * -0.75s, -0.25s, +0.25s, +0.75s (codes 0..3) with thresholds -s/2, 0,
 * +s/2, a value on a threshold taking the upper level.
 *   k_cache [B, Hkv, Cap, D] dtype (read), ctx_len [B] (read)
 *   block   power of two in [16, 256], Cap % block == 0
 *   codes   [B, Hkv, Cap, D/4] uint8 (written): channel c of a token is
 *           bits 2*(c%4) of byte c/4
 *   scales  [B, Hkv, Cap/block, D] dtype (written; exact, since max|k| is
 *           a key magnitude)
 * Only blocks that are complete (all positions < ctx_len[b]) are written.
 */
sls_status sls_thumb_build(const sls_attn_desc* desc, const void* k_cache,
                           const int32_t* ctx_len, int32_t block,
                           uint8_t* codes, void* scales, void* stream);

/*
 * Quantise the block that the key at position pos[b] completes, if any
 * (pos[b] % block == block - 1).  pos[b] < 0 skips sequence b.  Same
 * layouts as sls_thumb_build.
 */
sls_status sls_thumb_update(const sls_attn_desc* desc, const void* k_cache,
                            const int32_t* pos, int32_t block,
                            uint8_t* codes, void* scales, void* stream);

/*
 * Thumbnails plus 8-bit residuals ("Faster Than Flash", Methodology 1: the
 * key splits into the 2-bit thumbnail and an 8-bit residual that recovers
 * the precision the thumbnail drops).  The codes and scales are those of
 * sls_thumb_build; the residual of element (t, c) is
 *   r = clamp(rint(((k - k^) * 508) / s), -127, 127),   0 when s == 0,
 * each step one IEEE float32 operation (k^ = (code - 1.5) * s / 2 exactly),
 * so that the refined key k~ = k^ + r * s / 508 is within s / 1016 of k.
 *   res  [B, Hkv, Cap, D] int8 (written for complete blocks only)
 * The _update form quantises the block that position pos[b] completes, as
 * sls_thumb_update does.  Errors: SLS_EINVAL for a null pointer or a block
 * that is not a power of two in [16, 256] dividing Cap.
 */
sls_status sls_thumb_residual_build(const sls_attn_desc* desc, const void* k_cache,
                                    const int32_t* ctx_len, int32_t block, uint8_t* codes,
                                    void* scales, int8_t* res, void* stream);
sls_status sls_thumb_residual_update(const sls_attn_desc* desc, const void* k_cache,
                                     const int32_t* pos, int32_t block, uint8_t* codes,
                                     void* scales, int8_t* res, void* stream);

/* ---- selection --------------------------------------------------------- */

/*
 * Quest page selection with a fixed budget ("Don't read the haystack",
 * Part two): for every (b, kv head) row and query head g of its group,
 * U[g,p] = sum_c max(q[g,c]*kmin[p,c], q[g,c]*kmax[p,c]); the row's page
 * score is max_g U[g,p] (one list per KV head, shared by its query heads).
 * Forced pages: the first n_sink_pages pages and every page holding one of
 * the last n_local_tokens positions.  The list holds the forced pages plus
 * the top (k - #forced) other pages by score, ties to the lower page
 * index, sorted ascending.  When the row has <= k pages all of them are
 * listed and the rest of the list is -1.
 *   q        [B, Hq, D] dtype (read)
 *   kmin     [B, Hkv, Cap/P, D] dtype (read); kmax likewise.  With P == 1
 *            a page is one token, its min and max are the key itself:
 *            pass the K cache as kmin and kmax == kmin (read once).
 *   ctx_len  [B] int32 (read)
 *   k        budget in pages, 1 <= k <= Cap/P, and k must cover the forced
 *            pages: k >= n_sink_pages + ceil(n_local_tokens/P) + 1
 *   page_idx [B*Hkv, k] int32 (written)
 *   workspace >= sls_select_pages_workspace_size() bytes of device memory
 *            (one 32-bit key per page of every row, and for rows of more
 *            than 8192 pages the candidates of the scoring CTAs: 12.5 more
 *            bytes per page; contents on entry are ignored and on exit
 *            unspecified)
 * The score is computed in fp32; two pages whose scores differ by less
 * than the fp32 rounding of the sum may rank either way.  Rows may hold at
 * most 262144 pages (Cap/P); larger capacities return SLS_EUNSUPPORTED.
 */
sls_status sls_select_pages(const sls_attn_desc* desc, const void* q,
                            const void* kmin, const void* kmax,
                            const int32_t* ctx_len, int32_t k,
                            int32_t n_sink_pages, int32_t n_local_tokens,
                            int32_t* page_idx, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Bytes of workspace sls_select_pages needs for this descriptor (0 if the
 * descriptor is invalid). */
size_t sls_select_pages_workspace_size(const sls_attn_desc* desc);

/*
 * sls_select_pages without a workspace argument, for callers that cannot
 * allocate device memory for one (for example a plugin whose host framework
 * only passes it input and output tensors, or a process whose memory is all
 * reserved up front so that a cudaMalloc during decoding would fail or stall
 * the device).  It is not an operation of the source pages: only the origin
 * of the scratch differs.  The per-page keys go to a 4 MiB array compiled
 * into the library (held on every device that loads it, until exit) instead
 * of a caller buffer; the call allocates nothing.
 *   Arguments, results and validation: as sls_select_pages.
 *   Shapes whose keys need more than 4 MiB (sls_select_pages_workspace_size)
 *   return SLS_EWORKSPACE and enqueue nothing.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before capturing a stream.  The address is cached with the id of the
 *   device's CUDA context: after a cudaDeviceReset (a new context, the
 *   array at a new address) the next call looks it up again, so make that
 *   call outside stream capture too.
 *   All calls share the array: calls whose kernels may overlap on the GPU
 *   (other streams, other host threads) race on it and must be serialised
 *   by the caller.  No part of it needs to be zero.
 */
sls_status sls_select_pages_static(const sls_attn_desc* desc, const void* q,
                                   const void* kmin, const void* kmax,
                                   const int32_t* ctx_len, int32_t k,
                                   int32_t n_sink_pages, int32_t n_local_tokens,
                                   int32_t* page_idx, void* stream);

/* Bytes of workspace sls_select_delta needs for this descriptor/block. */
size_t sls_select_delta_workspace_size(const sls_attn_desc* desc, int32_t block);

/*
 * Top-delta block selection over 2-bit thumbnails ("Faster Than Flash",
 * Methodology 2, eqs. 1-3, with eq. 4's 1/sqrt(d) scaling):
 *   m~[g]  = max over the tokens of block 0 and of the newest block
 *            (partial or not) of the exact score scale * q[g] . k
 *   a complete block b other than those two is kept when
 *            max_g max_{t in b} (scale * q[g] . k^[t] - m~[g]) >= -delta
 *            with k^ the thumbnail levels;
 *   block 0 and the newest block are always kept.
 * Output: count[r] kept blocks, block_idx[r, 0..count[r]) the kept block
 * numbers ascending (entries past count[r] are unspecified).
 *   q [B, Hq, D], k_cache [B, Hkv, Cap, D], codes/scales as written by
 *   sls_thumb_build with the same block; ctx_len [B]
 *   idx_stride >= Cap/block
 *   workspace  >= sls_select_delta_workspace_size() bytes
 * Scores are computed in fp32.
 */
sls_status sls_select_delta(const sls_attn_desc* desc, const void* q,
                            const void* k_cache, const uint8_t* codes,
                            const void* scales, const int32_t* ctx_len,
                            int32_t block, float delta, int32_t* count,
                            int32_t* block_idx, int32_t idx_stride,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/* ---- attention --------------------------------------------------------- */

/*
 * Split-K sparse decode attention, stage one of two-stage flash-decoding
 * ("Don't read the haystack", Part one; the sparse twin of Part two walks
 * a page list instead of a range).  For every row r = (b, h), the page list
 * page_idx[r*idx_stride + i], i < n_r (n_r = count[r] if count != NULL,
 * else k_fixed) is cut into num_splits contiguous slices; slice s of every
 * query head g of the group produces
 *   m = max x, l = sum exp(x - m), acc = sum exp(x - m) v
 * over the valid tokens of its pages (position < ctx_len[b]), with
 * x = scale * q.k.  The sink is NOT applied here (see combine).
 * page_idx == NULL attends every page 0..ceil(ctx_len/P)-1 (dense decode).
 *   q [B, Hq, D], k_cache/v_cache [B, Hkv, Cap, D] dtype (read)
 *   o_part [B, Hq, num_splits, D] f32, m_part/l_part [B, Hq, num_splits]
 *   f32 (written; m in natural-log units; an empty slice gives m = -inf,
 *   l = 0, acc = 0)
 *   1 <= num_splits <= 1024
 */
sls_status sls_sparse_decode_attend(const sls_attn_desc* desc, const void* q,
                                    const void* k_cache, const void* v_cache,
                                    const int32_t* page_idx, int32_t idx_stride,
                                    const int32_t* count, int32_t k_fixed,
                                    const int32_t* ctx_len, int32_t num_splits,
                                    float* o_part, float* m_part, float* l_part,
                                    void* stream);

/*
 * Stage two: merge the splits with the log-sum-exp rescale ("Don't read the
 * haystack", Part one) and fold in the optional per-query-head sink as a
 * virtual key with value 0 ("Training-free sparse attention for
 * long-context LLM decode", section 1): with M = max(max_s m_s, sink_h),
 *   L = sum_s l_s e^(m_s - M) + e^(sink_h - M),
 *   out = sum_s acc_s e^(m_s - M) / L,   lse = M + log L.
 * The sink is a raw logit (not scaled).  Rows with no token and no sink
 * give out = 0, lse = -inf.
 *   o_part/m_part/l_part as written by sls_sparse_decode_attend
 *   sink [Hq] f32 or NULL
 *   out [B, Hq, D] dtype (written); lse [B, Hq] f32 or NULL (written)
 */
sls_status sls_combine_splits(const sls_attn_desc* desc, const float* o_part,
                              const float* m_part, const float* l_part,
                              int32_t num_splits, const float* sink, void* out,
                              float* lse, void* stream);

/*
 * A split count for sls_sparse_decode_attend(_combine) that gives about two
 * waves of CTAs on this GPU, each slice holding at least 64 tokens of a
 * list of up to max_entries pages.  Returns 1 for an invalid descriptor.
 */
int32_t sls_attend_default_splits(const sls_attn_desc* desc, int32_t max_entries);

/* Bytes of workspace sls_sparse_decode_attend_combine needs (num_splits 0:
 * the library's own schedule on the current device). */
size_t sls_attend_combine_workspace_size(const sls_attn_desc* desc,
                                         int32_t num_splits);

/*
 * Both stages in one launch: sls_sparse_decode_attend followed, inside the
 * same kernel, by the combine of each row.  num_splits == 0 lets the library
 * pick the split count (sls_attend_default_splits).  Where the tensor-map
 * fed kernel runs (bf16, pages of >= 16 tokens) with at most 16 splits, the
 * splits of a row form one thread-block cluster and combine through
 * distributed shared memory; otherwise every CTA of a row takes an arrival
 * ticket after writing its partials and the CTA that arrives last merges the
 * row's splits exactly as sls_combine_splits does (no CTA ever waits for
 * another).  Arguments as in the two separate calls; the partials live in
 * the workspace, whose first 4*B*Hkv bytes hold the tickets.
 *   workspace  >= sls_attend_combine_workspace_size() bytes; it must be
 *              zero-filled before its first use, and every call leaves the
 *              tickets at zero again.  Calls sharing a workspace must not
 *              run concurrently.
 */
sls_status sls_sparse_decode_attend_combine(const sls_attn_desc* desc, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            const int32_t* page_idx, int32_t idx_stride,
                                            const int32_t* count, int32_t k_fixed,
                                            const int32_t* ctx_len, int32_t num_splits,
                                            const float* sink, void* out, float* lse,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream);

/*
 * Refined top-delta attention ("Faster Than Flash", Methodology 3 step 3,
 * eq. 4): attention over each row's kept blocks in which the tokens of
 * complete blocks are scored with the refined key
 *   k~ = (code - 1.5) * s / 2 + r * s / 508
 * (thumbnail level plus 8-bit residual, sls_thumb_residual_build) instead
 * of the bf16 key; tokens of the newest, partial block are scored with the
 * bf16 key.  Values are the bf16 V.  With codes, scales and res all NULL
 * every token is scored with its bf16 key (plain attention over the lists).
 * The rows' lists, of different lengths, are cut into work items of equal
 * length spread over the GPU; each row's last item merges the row (sink,
 * lse as in sls_combine_splits).
 *   desc.page_size  the thumbnail block (>= 16); bf16, G <= 8, D 64 or 128,
 *                   B*Hkv <= 4096
 *   codes, scales, res  as written by sls_thumb_residual_build/_update
 *   block_idx [B*Hkv, idx_stride] int32, count [B*Hkv] int32: the kept
 *             blocks of each row (sls_select_delta's output); -1 entries
 *             and blocks past the context are skipped
 *   workspace >= sls_refined_decode_attend_workspace_size() bytes, zero-
 *             filled before its first use (every call leaves its arrival
 *             counters at zero); calls sharing it must not run concurrently
 *   |q * s| must stay below 65504 (the products run in fp16 hi/lo parts).
 * Errors: SLS_EUNSUPPORTED for another dtype, G > 8, blocks < 16 tokens or
 * more rows; SLS_EINVAL for null or misaligned pointers or bad sizes;
 * SLS_EWORKSPACE.
 */
size_t sls_refined_decode_attend_workspace_size(const sls_attn_desc* desc);
sls_status sls_refined_decode_attend_combine(const sls_attn_desc* desc, const void* q,
                                             const void* k_cache, const void* v_cache,
                                             const uint8_t* codes, const void* scales,
                                             const int8_t* res, const int32_t* block_idx,
                                             int32_t idx_stride, const int32_t* count,
                                             const int32_t* ctx_len, const float* sink,
                                             void* out, float* lse, void* workspace,
                                             size_t workspace_bytes, void* stream);

/* ---- the whole Quest decode step ---------------------------------------- */

/* Bytes of workspace sls_quest_decode_step needs for this budget and split
 * count (0 on an invalid descriptor). */
size_t sls_quest_decode_step_workspace_size(const sls_attn_desc* desc, int32_t k, int32_t num_splits);

/* CTAs per row (the cluster size) the one-launch Quest step uses for this
 * shape and budget by default; 0 when the shape takes the two-launch path. */
int32_t sls_quest_decode_step_splits(const sls_attn_desc* desc, int32_t k);

/*
 * One Quest decode step: the selection of sls_select_pages (budget k,
 * n_sink_pages, n_local_tokens, same tie rule and list order) and the
 * sparse attention with the combine of sls_sparse_decode_attend_combine
 * over the chosen pages ("Don't read the haystack", Part two).
 *
 * For bf16 caches with pages of >= 16 tokens (k <= 4096, Cap/P <= 131072)
 * this is ONE kernel launch: a
 * thread-block cluster per (sequence, KV head) scores its row's pages from
 * the min/max metadata, selects the top k inside the cluster and attends to
 * them; the scores and the page list never leave shared memory.  Otherwise
 * the call runs sls_select_pages then sls_sparse_decode_attend_combine.
 *   kmin, kmax  [B, Hkv, Cap/P, D] page metadata (sls_pagemeta_build)
 *   page_idx    [B*Hkv, k] int32 receiving the chosen pages (ascending, -1
 *               padded), or NULL
 *   out, lse    as in sls_combine_splits
 *   num_splits  CTAs per row (0: the library's choice; the one-launch kernel
 *               uses at most 16)
 *   min_sparsity  sparsity gate ("perf(core): fused sparse-attention decode
 *               via page indirection", Corrected premise 2): a row whose
 *               context holds fewer than min_sparsity * k * P tokens is
 *               attended densely over its whole context, without selection,
 *               and its page_idx row is left at -1.  0 disables the gate.
 *               The gate needs the one-launch kernel: on the two-launch path
 *               a non-zero value returns SLS_EUNSUPPORTED.
 *   workspace   >= sls_quest_decode_step_workspace_size() bytes, zero-filled
 *               before its first use (the one-launch kernel leaves it alone;
 *               the two-launch path keeps its tickets at zero).
 */
sls_status sls_quest_decode_step(const sls_attn_desc* desc, const void* q, const void* k_cache,
                                 const void* v_cache, const void* kmin, const void* kmax,
                                 const int32_t* ctx_len, int32_t k, int32_t n_sink_pages,
                                 int32_t n_local_tokens, const float* sink, int32_t* page_idx,
                                 void* out, float* lse, int32_t num_splits, float min_sparsity,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* ---- selection quality ------------------------------------------------- */

/* Bytes of workspace sls_selection_recall needs. */
size_t sls_selection_recall_workspace_size(const sls_attn_desc* desc);

/*
 * Attention-mass recall of page lists ("Don't read the haystack", Part
 * three: how much of the true attention mass the selected pages hold): for
 * every query head, the share of its full-context softmax mass (scores
 * scale * q.k over the positions < ctx_len; no sink) that falls on the
 * tokens of its row's listed pages.  A diagnostic beside the decode step: it
 * reads every key of the context.
 *   page_idx, idx_stride, count, k_fixed   as in sls_sparse_decode_attend
 *               (NULL page_idx: every page, recall 1)
 *   recall      [B, Hq] float; an empty context gives 1 (no mass missed)
 *   workspace   >= sls_selection_recall_workspace_size() bytes
 * Capacities above 262144 pages per row return SLS_EUNSUPPORTED.
 */
sls_status sls_selection_recall(const sls_attn_desc* desc, const void* q, const void* k_cache,
                                const int32_t* page_idx, int32_t idx_stride, const int32_t* count,
                                int32_t k_fixed, const int32_t* ctx_len, float* recall, void* workspace,
                                size_t workspace_bytes, void* stream);

/* ---- diagnostics ------------------------------------------------------- */

/* Message of the last failing call on this thread ("" if none). */
const char* sls_last_error(void);

/*
 * Device status of the kernels since the previous check ("perf(core): fused
 * sparse-attention decode via page indirection", Making the selection
 * inspectable: every call has an observable outcome).  Two kinds of events
 * are counted on the device:
 *   - a bounded wait on a copy pipeline that gave up (kernels that stage data
 *     through shared memory poll their copies a bounded number of times; the
 *     affected outputs become NaN);
 *   - a page-list entry that is neither a page of the pool [0, Cap/P) nor the
 *     -1 padding (the attend and recall kernels skip it: it gives no token).
 * This call synchronises the device, reads and clears the counts (one atomic
 * exchange per word, so no count is lost), and returns SLS_ETIMEOUT if any
 * wait gave up, else SLS_EDEVICE if any bad entry was met, else SLS_OK
 * (SLS_ECUDA if the device cannot be read); the message gives the counts.
 * The counts are global to the process: they cover every launch since the
 * previous check, on every stream and host thread, so only calls ordered
 * with the check are attributed to it.
 */
sls_status sls_pipeline_check(void);

/*
 * Which paths the library took ("perf(core): fused sparse-attention decode
 * via page indirection", Proving which path a benchmark arm took: a
 * benchmark must be able to show which kernel it measured).  Host counters
 * count launches by the kernel the library picked; the two row counters are
 * kept on the device by the one-launch step.
 */
typedef struct sls_stats {
  uint64_t quest_step_one_launch;     /* sls_quest_decode_step calls run as one kernel */
  uint64_t quest_step_two_launch;     /* ... run as select + attend (shape outside the kernel) */
  uint64_t step_rows_dense;           /* rows the sparsity gate sent to dense attention */
  uint64_t step_rows_all_keys;        /* rows whose cluster selected from all of the row's keys
                                         (long rows, or the candidate check failed) */
  uint64_t select_pages;              /* sls_select_pages(_static) launches */
  uint64_t select_delta_tensor_cores; /* top-delta scans on the tensor cores */
  uint64_t select_delta_cuda_cores;   /* ... on the CUDA cores (fp32, or the CUDA-core flag) */
  uint64_t attend_tma;                /* split-K attends by kernel: tensor-map fed, */
  uint64_t attend_mma;                /* register-fed tensor cores, */
  uint64_t attend_cuda_cores;         /* CUDA cores */
  uint64_t attend_stream_k;           /* stream-K attends over block lists with bf16 keys */
  uint64_t attend_refined;            /* ... with the refined (2-bit + 8-bit) keys */
  uint64_t combine;                   /* separate combine launches */
  uint64_t metadata;                  /* page min/max, thumbnail, residual and append launches */
  uint64_t recall;                    /* selection-recall launches */
  uint64_t select_rows_all_keys;      /* rows wider than 8192 pages whose sls_select_pages top-k
                                         ranked all of the row's keys (the candidate check failed) */
  uint64_t attend_stream_k_tma;       /* of attend_stream_k: the tensor-map fed kernel */
  uint64_t attend_refined_tma;        /* of attend_refined: the tensor-map fed kernel */
} sls_stats;

/* Fills *out with the counters (synchronising the device to read the row
 * counters); reset != 0 zeroes them.  SLS_EINVAL for a NULL out. */
sls_status sls_get_stats(sls_stats* out, int32_t reset);

/* Library ABI version (major*10000 + minor*100 + patch). */
int32_t sls_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SLS_H */
