// C ABI of libsls: host-side validation, then launch.  Nothing here touches
// device memory or synchronises; a failed check returns before any launch.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "launch.h"
#include "sls.h"

namespace {

thread_local char g_err[512] = "";
std::atomic<unsigned long long> g_stats[sls::kStatCount];

sls_status fail(sls_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

sls_status ok() {
  g_err[0] = '\0';
  return SLS_OK;
}

sls_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(SLS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

// a*b*... with overflow detection against int64 and against the int32
// indexing the kernels use for per-row positions.
bool checked_mul(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

sls_status check_desc(const sls_attn_desc* d, sls::Shape* s) {
  if (!d) return fail(SLS_EINVAL, "desc is NULL");
  if (d->batch < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1)
    return fail(SLS_EINVAL, "batch/heads must be >= 1 (B=%d Hq=%d Hkv=%d)", d->batch,
                d->num_q_heads, d->num_kv_heads);
  if (d->num_q_heads % d->num_kv_heads)
    return fail(SLS_EINVAL, "num_q_heads %d not a multiple of num_kv_heads %d", d->num_q_heads,
                d->num_kv_heads);
  const int G = d->num_q_heads / d->num_kv_heads;
  if (G > 8) return fail(SLS_EUNSUPPORTED, "query heads per kv head G=%d > 8", G);
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(SLS_EUNSUPPORTED, "head_dim %d not in {64, 128}", d->head_dim);
  if (d->dtype != SLS_DTYPE_F32 && d->dtype != SLS_DTYPE_BF16)
    return fail(SLS_EUNSUPPORTED, "dtype %d", d->dtype);
  if (!pow2(d->page_size) || d->page_size > 256)
    return fail(SLS_EINVAL, "page_size %d must be a power of two in [1, 256]", d->page_size);
  if (d->capacity < 1 || d->capacity % d->page_size)
    return fail(SLS_EINVAL, "capacity %d must be >= 1 and a multiple of page_size %d", d->capacity,
                d->page_size);
  if (!(d->scale >= 0.f) || std::isinf(d->scale)) return fail(SLS_EINVAL, "scale must be finite and >= 0");
  if (d->flags & ~(SLS_FLAG_CUDA_CORES | SLS_FLAG_NO_TMA | SLS_FLAG_TEST_WAIT_TIMEOUT))
    return fail(SLS_EINVAL, "unknown flags 0x%x", d->flags);
  // element counts of the caches and of the per-row index space
  int64_t rows, elems;
  if (!checked_mul(d->batch, d->num_kv_heads, &rows) || !checked_mul(rows, d->capacity, &elems) ||
      !checked_mul(elems, d->head_dim, &elems) || rows > INT32_MAX || elems > (int64_t(1) << 48) ||
      (int64_t)d->batch * d->num_q_heads > INT32_MAX)
    return fail(SLS_EOVERFLOW, "cache size overflows");
  s->B = d->batch;
  s->Hq = d->num_q_heads;
  s->Hkv = d->num_kv_heads;
  s->G = G;
  s->D = d->head_dim;
  s->P = d->page_size;
  s->pshift = __builtin_ctz((unsigned)d->page_size);
  s->Cap = d->capacity;
  s->dtype = d->dtype;
  s->flags = d->flags;
  s->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->head_dim);
  return SLS_OK;
}

}  // namespace

namespace sls {
void stat_add(StatId id) { g_stats[id].fetch_add(1, std::memory_order_relaxed); }
}  // namespace sls

namespace sls {
// Records a failure message for sls_last_error() from another translation unit.
sls_status record_error(sls_status code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace sls

namespace {

#define REQUIRE(ptr)                                     \
  do {                                                   \
    if (!(ptr)) return fail(SLS_EINVAL, "%s is NULL", #ptr); \
  } while (0)

// Tensors the kernels read or write in 16-byte vectors.
#define REQUIRE16(ptr)                                                                      \
  do {                                                                                      \
    if (!(ptr)) return fail(SLS_EINVAL, "%s is NULL", #ptr);                                \
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return fail(SLS_EINVAL, "%s is not 16-byte aligned", #ptr); \
  } while (0)

}  // namespace

extern "C" {

const char* sls_last_error(void) { return g_err; }

int32_t sls_version(void) { return 10000; }

sls_status sls_get_stats(sls_stats* out, int32_t reset) {
  if (!out) return fail(SLS_EINVAL, "out is NULL");
  std::memset(out, 0, sizeof(*out));
  auto take = [&](sls::StatId id) -> uint64_t {
    return reset ? g_stats[id].exchange(0) : g_stats[id].load();
  };
  out->quest_step_one_launch = take(sls::kStatStepOneLaunch);
  out->quest_step_two_launch = take(sls::kStatStepTwoLaunch);
  out->select_pages = take(sls::kStatSelectPages);
  out->select_delta_tensor_cores = take(sls::kStatDeltaTensorCores);
  out->select_delta_cuda_cores = take(sls::kStatDeltaCudaCores);
  out->attend_tma = take(sls::kStatAttendTma);
  out->attend_mma = take(sls::kStatAttendMma);
  out->attend_cuda_cores = take(sls::kStatAttendCudaCores);
  out->attend_stream_k = take(sls::kStatAttendStreamK);
  out->attend_refined = take(sls::kStatAttendRefined);
  out->combine = take(sls::kStatCombine);
  out->metadata = take(sls::kStatMetadata);
  out->recall = take(sls::kStatRecall);
  out->attend_stream_k_tma = take(sls::kStatAttendStreamKTma);
  out->attend_refined_tma = take(sls::kStatAttendRefinedTma);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(SLS_ECUDA, "device synchronisation failed");
  unsigned long long dense = 0, all_keys = 0;
  sls::take_step_row_stats(&dense, &all_keys, reset != 0);
  out->step_rows_dense = dense;
  out->step_rows_all_keys = all_keys;
  out->select_rows_all_keys = sls::take_select_rows_all_keys(reset != 0);
  return ok();
}

sls_status sls_pipeline_check(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(SLS_ECUDA, "device synchronisation failed");
  unsigned int timeouts = 0, bad = 0;
  for (auto take : {sls::take_status_attend_cc, sls::take_status_attend_mma, sls::take_status_attend_tma,
                    sls::take_status_attend_refined, sls::take_status_quest_step, sls::take_status_recall}) {
    const sls::DeviceStatus st = take();
    timeouts += st.wait_timeouts;
    bad += st.bad_page_ids;
  }
  if (cudaGetLastError() != cudaSuccess) return fail(SLS_ECUDA, "reading the device status words failed");
  if (timeouts)
    return fail(SLS_ETIMEOUT, "%u pipelined CTA(s) gave up waiting for their copies (%u bad page-list entries)",
                timeouts, bad);
  if (bad) return fail(SLS_EDEVICE, "%u page-list entries were neither a page of the pool nor -1 (skipped)", bad);
  return SLS_OK;
}

sls_status sls_pagemeta_build(const sls_attn_desc* desc, const void* k_cache, const int32_t* ctx_len,
                              void* kmin, void* kmax, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(k_cache); REQUIRE(ctx_len); REQUIRE16(kmin); REQUIRE16(kmax);
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_pagemeta_build(s, k_cache, ctx_len, kmin, kmax, (cudaStream_t)stream),
                     "sls_pagemeta_build");
}

sls_status sls_pagemeta_update(const sls_attn_desc* desc, const void* k_cache, const int32_t* pos,
                               void* kmin, void* kmax, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(k_cache); REQUIRE(pos); REQUIRE16(kmin); REQUIRE16(kmax);
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_pagemeta_update(s, k_cache, pos, kmin, kmax, (cudaStream_t)stream),
                     "sls_pagemeta_update");
}

static sls_status check_block(const sls::Shape& s, int32_t block) {
  if (!pow2(block) || block < 16 || block > 256)
    return fail(SLS_EINVAL, "block %d must be a power of two in [16, 256]", block);
  if (s.Cap % block) return fail(SLS_EINVAL, "capacity %d not a multiple of block %d", s.Cap, block);
  return SLS_OK;
}

sls_status sls_decode_append(const sls_attn_desc* desc, const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, void* kmin, void* kmax, int32_t* ctx_len, int32_t* pos_out,
                             void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(k_new); REQUIRE16(v_new); REQUIRE16(k_cache); REQUIRE16(v_cache); REQUIRE(ctx_len);
  if ((kmin == nullptr) != (kmax == nullptr)) return fail(SLS_EINVAL, "kmin and kmax: both or neither");
  if (kmin && s.P == 1) return fail(SLS_EINVAL, "page_size 1: the key cache is its own page metadata (pass NULL)");
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_decode_append(s, k_new, v_new, k_cache, v_cache, kmin, kmax, ctx_len, pos_out,
                                               (cudaStream_t)stream),
                     "sls_decode_append");
}

sls_status sls_thumb_build(const sls_attn_desc* desc, const void* k_cache, const int32_t* ctx_len,
                           int32_t block, uint8_t* codes, void* scales, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  if ((r = check_block(s, block))) return r;
  REQUIRE16(k_cache); REQUIRE(ctx_len); REQUIRE16(codes); REQUIRE16(scales);
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_thumb_build(s, k_cache, ctx_len, block, codes, scales, nullptr,
                                             (cudaStream_t)stream),
                     "sls_thumb_build");
}

sls_status sls_thumb_residual_build(const sls_attn_desc* desc, const void* k_cache, const int32_t* ctx_len,
                                    int32_t block, uint8_t* codes, void* scales, int8_t* res, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  if ((r = check_block(s, block))) return r;
  REQUIRE16(k_cache); REQUIRE(ctx_len); REQUIRE16(codes); REQUIRE16(scales); REQUIRE16(res);
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_thumb_build(s, k_cache, ctx_len, block, codes, scales, res, (cudaStream_t)stream),
                     "sls_thumb_residual_build");
}

sls_status sls_thumb_update(const sls_attn_desc* desc, const void* k_cache, const int32_t* pos,
                            int32_t block, uint8_t* codes, void* scales, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  if ((r = check_block(s, block))) return r;
  REQUIRE16(k_cache); REQUIRE(pos); REQUIRE16(codes); REQUIRE16(scales);
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_thumb_update(s, k_cache, pos, block, codes, scales, nullptr,
                                              (cudaStream_t)stream),
                     "sls_thumb_update");
}

sls_status sls_thumb_residual_update(const sls_attn_desc* desc, const void* k_cache, const int32_t* pos,
                                     int32_t block, uint8_t* codes, void* scales, int8_t* res, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  if ((r = check_block(s, block))) return r;
  REQUIRE16(k_cache); REQUIRE(pos); REQUIRE16(codes); REQUIRE16(scales); REQUIRE16(res);
  sls::stat_add(sls::kStatMetadata);
  return cuda_status(sls::launch_thumb_update(s, k_cache, pos, block, codes, scales, res, (cudaStream_t)stream),
                     "sls_thumb_residual_update");
}

size_t sls_select_pages_workspace_size(const sls_attn_desc* desc) {
  sls::Shape s;
  if (check_desc(desc, &s)) return 0;
  return sls::select_pages_workspace(s);
}

sls_status sls_select_pages(const sls_attn_desc* desc, const void* q, const void* kmin,
                            const void* kmax, const int32_t* ctx_len, int32_t k,
                            int32_t n_sink_pages, int32_t n_local_tokens, int32_t* page_idx,
                            void* workspace, size_t workspace_bytes, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(q); REQUIRE16(kmin); REQUIRE16(kmax); REQUIRE(ctx_len); REQUIRE(page_idx);
  const int npcap = s.Cap >> s.pshift;
  if (k < 1 || k > npcap) return fail(SLS_EINVAL, "k=%d must be in [1, Cap/P=%d]", k, npcap);
  if (n_sink_pages < 0 || n_local_tokens < 0)
    return fail(SLS_EINVAL, "n_sink_pages and n_local_tokens must be >= 0");
  const int64_t forced_max =
      (int64_t)n_sink_pages + (n_local_tokens > 0 ? ((int64_t)n_local_tokens + s.P - 1) / s.P + 1 : 0);
  if (forced_max > k)
    return fail(SLS_EINVAL, "budget k=%d cannot hold the forced pages (up to %lld)", k,
                (long long)forced_max);
  if (s.P == 1 && kmin != kmax)
    return fail(SLS_EINVAL, "page_size 1: pass the key cache as both kmin and kmax");
  if (npcap > sls::select_pages_max_pages())
    return fail(SLS_EUNSUPPORTED, "Cap/P=%d pages per row exceeds the supported %d", npcap,
                sls::select_pages_max_pages());
  const size_t need = sls::select_pages_workspace(s);
  if (!workspace || workspace_bytes < need)
    return fail(SLS_EWORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  sls::stat_add(sls::kStatSelectPages);
  return cuda_status(sls::launch_select_pages(s, q, kmin, kmax, ctx_len, k, n_sink_pages, n_local_tokens,
                                              page_idx, workspace, (cudaStream_t)stream),
                     "sls_select_pages");
}

size_t sls_select_delta_workspace_size(const sls_attn_desc* desc, int32_t block) {
  sls::Shape s;
  if (check_desc(desc, &s) || check_block(s, block)) return 0;
  return sls::select_delta_workspace(s, block);
}

sls_status sls_select_delta(const sls_attn_desc* desc, const void* q, const void* k_cache,
                            const uint8_t* codes, const void* scales, const int32_t* ctx_len,
                            int32_t block, float delta, int32_t* count, int32_t* block_idx,
                            int32_t idx_stride, void* workspace, size_t workspace_bytes,
                            void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  if ((r = check_block(s, block))) return r;
  REQUIRE16(q); REQUIRE16(k_cache); REQUIRE16(codes); REQUIRE16(scales); REQUIRE(ctx_len);
  REQUIRE(count); REQUIRE(block_idx);
  if (!(delta >= 0.f) || std::isinf(delta)) return fail(SLS_EINVAL, "delta must be finite and >= 0");
  if (idx_stride < s.Cap / block)
    return fail(SLS_EINVAL, "idx_stride %d < Cap/block %d", idx_stride, s.Cap / block);
  const size_t need = sls::select_delta_workspace(s, block);
  if (!workspace || workspace_bytes < need)
    return fail(SLS_EWORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  return cuda_status(sls::launch_select_delta(s, q, k_cache, codes, scales, ctx_len, block, delta, count,
                                              block_idx, idx_stride, workspace, (cudaStream_t)stream),
                     "sls_select_delta");
}

sls_status sls_sparse_decode_attend(const sls_attn_desc* desc, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* page_idx, int32_t idx_stride,
                                    const int32_t* count, int32_t k_fixed, const int32_t* ctx_len,
                                    int32_t num_splits, float* o_part, float* m_part, float* l_part,
                                    void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(q); REQUIRE16(k_cache); REQUIRE16(v_cache); REQUIRE(ctx_len);
  REQUIRE16(o_part); REQUIRE(m_part); REQUIRE(l_part);
  if (num_splits < 1 || num_splits > 1024) return fail(SLS_EINVAL, "num_splits %d not in [1, 1024]", num_splits);
  if (page_idx) {
    if (idx_stride < 1) return fail(SLS_EINVAL, "idx_stride %d < 1", idx_stride);
    if (!count && (k_fixed < 0 || k_fixed > idx_stride))
      return fail(SLS_EINVAL, "k_fixed %d not in [0, idx_stride=%d]", k_fixed, idx_stride);
  }
  int64_t ctas;
  if (!checked_mul((int64_t)s.B * s.Hkv, num_splits, &ctas) || ctas > INT32_MAX)
    return fail(SLS_EOVERFLOW, "grid too large");
  return cuda_status(sls::launch_attend(s, q, k_cache, v_cache, page_idx, idx_stride, count, k_fixed, ctx_len,
                                        num_splits, o_part, m_part, l_part, (cudaStream_t)stream),
                     "sls_sparse_decode_attend");
}

int32_t sls_attend_default_splits(const sls_attn_desc* desc, int32_t max_entries) {
  sls::Shape s;
  if (check_desc(desc, &s) || max_entries < 1) return 1;
  return sls::attend_default_splits(s, max_entries);
}

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t sls_attend_combine_workspace_size(const sls_attn_desc* desc, int32_t num_splits) {
  sls::Shape s;
  if (check_desc(desc, &s) || num_splits < 0 || num_splits > 1024) return 0;
  if (num_splits == 0) num_splits = sls::max_auto_splits(s);
  const size_t heads = (size_t)s.B * s.Hq * num_splits;
  return align256((size_t)s.B * s.Hkv * 4) + align256(heads * s.D * 4) + 2 * align256(heads * 4);
}

sls_status sls_sparse_decode_attend_combine(const sls_attn_desc* desc, const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* page_idx, int32_t idx_stride,
                                            const int32_t* count, int32_t k_fixed, const int32_t* ctx_len,
                                            int32_t num_splits, const float* sink, void* out, float* lse,
                                            void* workspace, size_t workspace_bytes, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(q); REQUIRE16(k_cache); REQUIRE16(v_cache); REQUIRE(ctx_len); REQUIRE(out);
  if (num_splits < 0 || num_splits > 1024) return fail(SLS_EINVAL, "num_splits %d not in [0, 1024]", num_splits);
  if (page_idx) {
    if (idx_stride < 1) return fail(SLS_EINVAL, "idx_stride %d < 1", idx_stride);
    if (!count && (k_fixed < 0 || k_fixed > idx_stride))
      return fail(SLS_EINVAL, "k_fixed %d not in [0, idx_stride=%d]", k_fixed, idx_stride);
  }
  int64_t ctas;
  if (!checked_mul((int64_t)s.B * s.Hkv, num_splits, &ctas) || ctas > INT32_MAX)
    return fail(SLS_EOVERFLOW, "grid too large");
  const size_t need = sls_attend_combine_workspace_size(desc, num_splits);
  if (!workspace || workspace_bytes < need)
    return fail(SLS_EWORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  char* w = static_cast<char*>(workspace);
  const size_t heads = (size_t)s.B * s.Hq * (num_splits ? num_splits : sls::max_auto_splits(s));
  sls::FusedCombine f;
  f.tickets = reinterpret_cast<int32_t*>(w);
  w += align256((size_t)s.B * s.Hkv * 4);
  float* o_part = reinterpret_cast<float*>(w);
  w += align256(heads * s.D * 4);
  float* m_part = reinterpret_cast<float*>(w);
  w += align256(heads * 4);
  float* l_part = reinterpret_cast<float*>(w);
  f.sink = sink;
  f.out = out;
  f.lse = lse;
  return cuda_status(sls::launch_attend(s, q, k_cache, v_cache, page_idx, idx_stride, count, k_fixed, ctx_len,
                                        num_splits, o_part, m_part, l_part, (cudaStream_t)stream, &f),
                     "sls_sparse_decode_attend_combine");
}

size_t sls_refined_decode_attend_workspace_size(const sls_attn_desc* desc) {
  sls::Shape s;
  if (check_desc(desc, &s)) return 0;
  return sls::refined_workspace(s);
}

sls_status sls_refined_decode_attend_combine(const sls_attn_desc* desc, const void* q, const void* k_cache,
                                             const void* v_cache, const uint8_t* codes, const void* scales,
                                             const int8_t* res, const int32_t* block_idx, int32_t idx_stride,
                                             const int32_t* count, const int32_t* ctx_len, const float* sink,
                                             void* out, float* lse, void* workspace, size_t workspace_bytes,
                                             void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(q); REQUIRE16(k_cache); REQUIRE16(v_cache); REQUIRE(block_idx); REQUIRE(count); REQUIRE(ctx_len);
  REQUIRE(out);
  if ((codes == nullptr) != (res == nullptr) || (codes == nullptr) != (scales == nullptr))
    return fail(SLS_EINVAL, "codes, scales and res: all or none");
  if (!sls::refined_supported(s))
    return fail(SLS_EUNSUPPORTED,
                "needs bf16, G <= 8, blocks (page_size) of >= 16 tokens and at most 4096 rows (B*Hkv)");
  if (idx_stride < 1) return fail(SLS_EINVAL, "idx_stride %d < 1", idx_stride);
  if (codes) {
    REQUIRE16(codes); REQUIRE16(scales); REQUIRE16(res);
  }
  const size_t need = sls::refined_workspace(s);
  if (!workspace || workspace_bytes < need)
    return fail(SLS_EWORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  sls::stat_add(codes ? sls::kStatAttendRefined : sls::kStatAttendStreamK);
  return cuda_status(sls::launch_attend_refined(s, q, k_cache, v_cache, codes, scales, res, block_idx, idx_stride,
                                                count, ctx_len, sink, out, lse, workspace, (cudaStream_t)stream),
                     "sls_refined_decode_attend_combine");
}

size_t sls_quest_decode_step_workspace_size(const sls_attn_desc* desc, int32_t k, int32_t num_splits) {
  sls::Shape s;
  if (check_desc(desc, &s) || k < 1 || num_splits < 0 || num_splits > 1024) return 0;
  // what the two-launch path needs (the one-launch kernel uses none of it)
  return align256(sls::select_pages_workspace(s)) + align256((size_t)s.B * s.Hkv * k * 4) +
         sls_attend_combine_workspace_size(desc, num_splits);
}

int32_t sls_quest_decode_step_splits(const sls_attn_desc* desc, int32_t k) {
  sls::Shape s;
  if (check_desc(desc, &s) || k < 1 || k > (s.Cap >> s.pshift) || !sls::quest_step_eligible(s, k)) return 0;
  return sls::quest_step_splits(s, k);
}

sls_status sls_quest_decode_step(const sls_attn_desc* desc, const void* q, const void* k_cache, const void* v_cache,
                                 const void* kmin, const void* kmax, const int32_t* ctx_len, int32_t k,
                                 int32_t n_sink_pages, int32_t n_local_tokens, const float* sink, int32_t* page_idx,
                                 void* out, float* lse, int32_t num_splits, float min_sparsity, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(q); REQUIRE16(k_cache); REQUIRE16(v_cache); REQUIRE16(kmin); REQUIRE16(kmax); REQUIRE(ctx_len); REQUIRE(out);
  const int npcap = s.Cap >> s.pshift;
  if (k < 1 || k > npcap) return fail(SLS_EINVAL, "k=%d must be in [1, Cap/P=%d]", k, npcap);
  if (n_sink_pages < 0 || n_local_tokens < 0) return fail(SLS_EINVAL, "n_sink_pages and n_local_tokens must be >= 0");
  const int64_t forced_max =
      (int64_t)n_sink_pages + (n_local_tokens > 0 ? ((int64_t)n_local_tokens + s.P - 1) / s.P + 1 : 0);
  if (forced_max > k)
    return fail(SLS_EINVAL, "budget k=%d cannot hold the forced pages (up to %lld)", k, (long long)forced_max);
  if (s.P == 1 && kmin != kmax) return fail(SLS_EINVAL, "page_size 1: pass the key cache as both kmin and kmax");
  if (num_splits < 0 || num_splits > 1024) return fail(SLS_EINVAL, "num_splits %d not in [0, 1024]", num_splits);
  if (!(min_sparsity >= 0.f) || std::isinf(min_sparsity))
    return fail(SLS_EINVAL, "min_sparsity must be finite and >= 0");
  const size_t need = sls_quest_decode_step_workspace_size(desc, k, num_splits);
  if (!workspace || workspace_bytes < need)
    return fail(SLS_EWORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  bool handled = false;
  cudaError_t e = sls::launch_quest_step(s, q, k_cache, v_cache, kmin, kmax, ctx_len, k, n_sink_pages,
                                         n_local_tokens, sink, page_idx, out, lse, num_splits, min_sparsity,
                                         (cudaStream_t)stream, &handled);
  if (handled) {
    sls::stat_add(sls::kStatStepOneLaunch);
    return cuda_status(e, "sls_quest_decode_step");
  }
  if (min_sparsity > 0.f)
    return fail(SLS_EUNSUPPORTED, "min_sparsity needs the one-launch step (bf16, pages of >= 16 tokens)");
  // two launches: select into page_idx (or the workspace), then attend with the fused combine
  sls::stat_add(sls::kStatStepTwoLaunch);
  if (npcap > sls::select_pages_max_pages())
    return fail(SLS_EUNSUPPORTED, "Cap/P=%d pages per row exceeds the supported %d", npcap,
                sls::select_pages_max_pages());
  char* w = static_cast<char*>(workspace);
  void* sel_ws = w;
  w += align256(sls::select_pages_workspace(s));
  int32_t* list = page_idx ? page_idx : reinterpret_cast<int32_t*>(w);
  w += align256((size_t)s.B * s.Hkv * k * 4);
  e = sls::launch_select_pages(s, q, kmin, kmax, ctx_len, k, n_sink_pages, n_local_tokens, list, sel_ws,
                               (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "sls_quest_decode_step (select)");
  const size_t heads = (size_t)s.B * s.Hq * (num_splits ? num_splits : sls::max_auto_splits(s));
  sls::FusedCombine f;
  f.tickets = reinterpret_cast<int32_t*>(w);
  w += align256((size_t)s.B * s.Hkv * 4);
  float* o_part = reinterpret_cast<float*>(w);
  w += align256(heads * s.D * 4);
  float* m_part = reinterpret_cast<float*>(w);
  w += align256(heads * 4);
  float* l_part = reinterpret_cast<float*>(w);
  f.sink = sink;
  f.out = out;
  f.lse = lse;
  return cuda_status(sls::launch_attend(s, q, k_cache, v_cache, list, k, nullptr, k, ctx_len, num_splits, o_part,
                                        m_part, l_part, (cudaStream_t)stream, &f),
                     "sls_quest_decode_step (attend)");
}

size_t sls_selection_recall_workspace_size(const sls_attn_desc* desc) {
  sls::Shape s;
  if (check_desc(desc, &s)) return 0;
  return sls::recall_workspace(s);
}

sls_status sls_selection_recall(const sls_attn_desc* desc, const void* q, const void* k_cache,
                                const int32_t* page_idx, int32_t idx_stride, const int32_t* count, int32_t k_fixed,
                                const int32_t* ctx_len, float* recall, void* workspace, size_t workspace_bytes,
                                void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(q); REQUIRE16(k_cache); REQUIRE(ctx_len); REQUIRE(recall);
  if (page_idx) {
    if (idx_stride < 1) return fail(SLS_EINVAL, "idx_stride %d < 1", idx_stride);
    if (!count && (k_fixed < 0 || k_fixed > idx_stride))
      return fail(SLS_EINVAL, "k_fixed %d not in [0, idx_stride=%d]", k_fixed, idx_stride);
  }
  if (!sls::recall_supported(s)) return fail(SLS_EUNSUPPORTED, "Cap/P above 262144 pages");
  const size_t need = sls::recall_workspace(s);
  if (!workspace || workspace_bytes < need)
    return fail(SLS_EWORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  sls::stat_add(sls::kStatRecall);
  return cuda_status(sls::launch_recall(s, q, k_cache, page_idx, idx_stride, count, k_fixed, ctx_len, recall,
                                        workspace, (cudaStream_t)stream),
                     "sls_selection_recall");
}

sls_status sls_combine_splits(const sls_attn_desc* desc, const float* o_part, const float* m_part,
                              const float* l_part, int32_t num_splits, const float* sink, void* out,
                              float* lse, void* stream) {
  sls::Shape s;
  sls_status r = check_desc(desc, &s);
  if (r) return r;
  REQUIRE16(o_part); REQUIRE(m_part); REQUIRE(l_part); REQUIRE(out);
  if (num_splits < 1 || num_splits > 1024) return fail(SLS_EINVAL, "num_splits %d not in [1, 1024]", num_splits);
  return cuda_status(sls::launch_combine(s, o_part, m_part, l_part, num_splits, sink, out, lse, (cudaStream_t)stream),
                     "sls_combine_splits");
}

}  // extern "C"
