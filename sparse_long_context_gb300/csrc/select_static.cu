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
//
// The array's device address is looked up on the first call on each device
// (that call should come before any stream capture) and cached with the id
// of the CUDA context it belongs to.  A device reset, or anything else that
// replaces the device's primary context, reloads the library's module at a
// new address; the next call sees a different context id and looks the
// address up again.
#include <cuda.h>

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
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the current CUDA context (unique for the life of the process), or 0
// when it cannot be read.
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  static const CtxGetIdFn get_id = []() -> CtxGetIdFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<CtxGetIdFn>(p);
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of this device's copy of the array.  The host-side name
// g_select_scratch is not a device address, so it is looked up with the
// device current and cached per device together with the context id; a
// changed id (a reset device) or an unreadable one looks it up again.
sls_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return sls::record_error(SLS_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return sls::record_error(SLS_EUNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch failed: %s", cudaGetErrorString(e));
      return sls::record_error(SLS_ECUDA, msg);
    }
    g_scratch_ptr[dev] = p;
    // the lookup made the device's primary context current if none was
    g_scratch_ctx[dev] = ctx ? ctx : current_context_id();
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
