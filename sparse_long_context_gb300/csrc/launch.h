// Internal (C++) launch interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments have been validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace sls {

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream drains; it waits for it in
// pdl_wait_then_release() before touching memory.
// With cluster > 1, consecutive groups of `cluster` CTAs along x form a
// thread-block cluster (grid.x must be a multiple of it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster,
                                      cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  return launch_pdl_cluster(kern, grid, block, smem, 1, st, std::forward<Args>(args)...);
}

// Descriptor flags (the public SLS_FLAG_* values).
constexpr int kFlagCudaCores = 1;
constexpr int kFlagNoTma = 2;
constexpr int kFlagTestWaitTimeout = 4;

struct Shape {
  int B, Hq, Hkv, G, D, P, pshift, Cap, dtype, flags;
  float scale;
};

cudaError_t launch_pagemeta_build(const Shape& s, const void* k, const int32_t* ctx_len,
                                  void* kmin, void* kmax, cudaStream_t st);
cudaError_t launch_pagemeta_update(const Shape& s, const void* k, const int32_t* pos,
                                   void* kmin, void* kmax, cudaStream_t st);
cudaError_t launch_decode_append(const Shape& s, const void* k_new, const void* v_new, void* k, void* v,
                                 void* kmin, void* kmax, int32_t* ctx_len, int32_t* pos_out, cudaStream_t st);
cudaError_t launch_thumb_build(const Shape& s, const void* k, const int32_t* ctx_len,
                               int block, uint8_t* codes, void* scales, int8_t* res, cudaStream_t st);
cudaError_t launch_thumb_update(const Shape& s, const void* k, const int32_t* pos,
                                int block, uint8_t* codes, void* scales, int8_t* res, cudaStream_t st);

bool refined_supported(const Shape& s);
size_t refined_workspace(const Shape& s);
cudaError_t launch_attend_refined(const Shape& s, const void* q, const void* k, const void* v, const uint8_t* codes,
                                  const void* scales, const int8_t* res, const int32_t* block_idx, int idx_stride,
                                  const int32_t* count, const int32_t* ctx_len, const float* sink, void* out,
                                  float* lse, void* ws, cudaStream_t st);

size_t select_pages_workspace(const Shape& s);
cudaError_t launch_select_pages(const Shape& s, const void* q, const void* kmin,
                                const void* kmax, const int32_t* ctx_len, int k,
                                int n_sink_pages, int n_local_tokens, int32_t* page_idx,
                                void* ws, cudaStream_t st);

size_t select_delta_workspace(const Shape& s, int block);
cudaError_t launch_select_delta(const Shape& s, const void* q, const void* k,
                                const uint8_t* codes, const void* scales,
                                const int32_t* ctx_len, int block, float delta,
                                int32_t* count, int32_t* block_idx, int idx_stride,
                                void* ws, cudaStream_t st);

struct FusedCombine {
  int32_t* tickets;
  const float* sink;
  void* out;
  float* lse;
};
int attend_default_splits(const Shape& s, int max_entries);
// Tensor-map fed attend kernel (bf16, pages of >= 16 tokens).
bool attend_tma_eligible(const Shape& s);
int attend_tma_per_sm(const Shape& s);
int attend_tma_splits(const Shape& s, int groups_per_row);
// Device status words of each translation unit whose kernels count them,
// read and cleared by take_status_<unit>() (see status.cuh).
struct DeviceStatus {
  unsigned int bad_page_ids;   // page-list entries that are neither a page of the pool nor the -1 padding
  unsigned int wait_timeouts;  // bounded waits on a copy pipeline that gave up
};
DeviceStatus take_status_attend_cc();
DeviceStatus take_status_attend_mma();
DeviceStatus take_status_attend_tma();
DeviceStatus take_status_attend_refined();
DeviceStatus take_status_quest_step();
DeviceStatus take_status_recall();

// Fused Quest step (bf16, pages of >= 16 tokens): select + attend + combine
// in one launch.  *handled is false (and nothing is enqueued) when the shape
// is not covered.
bool quest_step_eligible(const Shape& s, int k);
int quest_step_splits(const Shape& s, int k);
cudaError_t launch_quest_step(const Shape& s, const void* q, const void* k_cache, const void* v_cache,
                              const void* kmin, const void* kmax, const int32_t* ctx_len, int k, int n_sink,
                              int n_local, const float* sink, int32_t* page_idx, void* out, float* lse,
                              int num_splits, float min_sparsity, cudaStream_t st, bool* handled);

// Selection quality: attention-mass recall of page lists (a diagnostic).
size_t recall_workspace(const Shape& s);
bool recall_supported(const Shape& s);
cudaError_t launch_recall(const Shape& s, const void* q, const void* k, const int32_t* page_idx, int idx_stride,
                          const int32_t* count, int k_fixed, const int32_t* ctx_len, float* recall, void* ws,
                          cudaStream_t st);
int max_auto_splits(const Shape& s);
cudaError_t launch_attend(const Shape& s, const void* q, const void* k, const void* v,
                          const int32_t* page_idx, int idx_stride, const int32_t* count,
                          int k_fixed, const int32_t* ctx_len, int num_splits,
                          float* o_part, float* m_part, float* l_part, cudaStream_t st,
                          const FusedCombine* fused = nullptr);

cudaError_t launch_combine(const Shape& s, const float* o_part, const float* m_part,
                           const float* l_part, int num_splits, const float* sink,
                           void* out, float* lse, cudaStream_t st);

// Streaming multiprocessors of the current device (cached per device).
// Which paths the library took (read back by sls_get_stats): host counters
// bumped where a launch picks its kernel.
enum StatId {
  kStatStepOneLaunch, kStatStepTwoLaunch, kStatSelectPages, kStatDeltaTensorCores, kStatDeltaCudaCores,
  kStatAttendTma, kStatAttendMma, kStatAttendCudaCores, kStatAttendStreamK, kStatAttendRefined, kStatCombine,
  kStatMetadata, kStatRecall, kStatAttendStreamKTma, kStatAttendRefinedTma, kStatCount
};
void stat_add(StatId id);
// Rows the one-launch step attended densely (sparsity gate) and rows whose
// cluster selected from all of the row's keys, counted on the device.
void take_step_row_stats(unsigned long long* dense, unsigned long long* all_keys, bool reset);
// Wide rows of sls_select_pages whose top-k CTA selected from all keys.
unsigned long long take_select_rows_all_keys(bool reset);

inline int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
  return cache[dev] > 0 ? cache[dev] : 1;
}

// Most pages (Cap/P) a row of sls_select_pages may hold.
int select_pages_max_pages();

}  // namespace sls
