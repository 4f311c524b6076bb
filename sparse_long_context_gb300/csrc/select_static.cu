// sls_select_pages_static: Quest page selection for callers that cannot give
// the library a workspace.
//
// sls_select_pages needs a caller-provided device buffer for its per-page
// keys.  Some callers have no way to provide one: a plugin that its host
// framework only hands input and output tensors, or a process whose device
// memory is reserved up front by a caching allocator, where a cudaMalloc in
// the decode loop would fail or stall the whole device.  This entry point
// takes its key scratch from a fixed array compiled into the library
// instead, and allocates nothing.
//
// The array is kStaticScratchBytes (4 MiB) of device memory held by every
// GPU that loads the library, until the process exits.  Every call uses the
// same array, so two calls whose kernels overlap on the GPU (on different
// streams, or from different host threads) race on it and must be ordered
// by the caller.  Nothing in it has to start at zero: each call writes every
// key it later reads.
#include <cstdio>
#include <mutex>

#include "launch.h"
#include "sls.h"

namespace sls {
sls_status record_error(sls_status code, const char* msg);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of this device's copy of the array.  The host-side name
// g_select_scratch is not a device address, so it is looked up once per
// device (with that device current) and cached.
sls_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return sls::record_error(SLS_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return sls::record_error(SLS_EUNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch failed: %s", cudaGetErrorString(e));
      return sls::record_error(SLS_ECUDA, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SLS_OK;
}

}  // namespace

extern "C" sls_status sls_select_pages_static(const sls_attn_desc* desc, const void* q, const void* kmin,
                                              const void* kmax, const int32_t* ctx_len, int32_t k,
                                              int32_t n_sink_pages, int32_t n_local_tokens,
                                              int32_t* page_idx, void* stream) {
  const size_t need = sls_select_pages_workspace_size(desc);
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "sls_select_pages_static: this shape needs %zu bytes of scratch, the built-in scratch holds %zu; "
             "use sls_select_pages with a workspace",
             need, kStaticScratchBytes);
    return sls::record_error(SLS_EWORKSPACE, msg);
  }
  void* scratch = nullptr;
  const sls_status st = scratch_for_current_device(&scratch);
  if (st != SLS_OK) return st;
  // same validation and kernels as sls_select_pages, scratch from the array
  return sls_select_pages(desc, q, kmin, kmax, ctx_len, k, n_sink_pages, n_local_tokens, page_idx, scratch,
                          kStaticScratchBytes, stream);
}
