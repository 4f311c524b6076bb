// Device status words: what a kernel could not do, counted on the device and
// read back by the host (sls_pipeline_check).
//
// The library is built without relocatable device code, so every translation
// unit that includes this header has its own copy of the counters and its own
// take_status_here(); api.cu adds up the copies of the units whose kernels
// count.  The host reads and clears a copy with one atomic exchange per word
// (a one-thread kernel), so a count that lands between the read and the clear
// is not lost.  The words are global to the process: a check reports every
// count since the previous check, from any stream or host thread.
#pragma once

#include <cuda_runtime.h>

#include "launch.h"

namespace sls {

static __device__ DeviceStatus g_status = {0u, 0u};
static __device__ DeviceStatus g_status_taken = {0u, 0u};

// A page-list entry is bad when it is neither the -1 padding nor a page of
// the pool [0, npages).  Such entries are skipped (they contribute no token).
__device__ __forceinline__ bool bad_page_id(int pg, int npages) {
  return pg != -1 && (unsigned)pg >= (unsigned)npages;
}
__device__ __forceinline__ void note_bad_pages(unsigned int n) {
  if (n) atomicAdd(&g_status.bad_page_ids, n);
}
__device__ __forceinline__ void note_wait_timeout() { atomicAdd(&g_status.wait_timeouts, 1u); }

static __global__ void take_status_kernel() {
  g_status_taken.bad_page_ids = atomicExch(&g_status.bad_page_ids, 0u);
  g_status_taken.wait_timeouts = atomicExch(&g_status.wait_timeouts, 0u);
}

// Reads and clears this unit's counters (on the legacy default stream, which
// orders it after the caller's synchronisation).  Zero counts if the device
// cannot be read.
static inline DeviceStatus take_status_here() {
  DeviceStatus v = {0u, 0u};
  take_status_kernel<<<1, 1>>>();
  if (cudaGetLastError() != cudaSuccess) return v;
  if (cudaMemcpyFromSymbol(&v, g_status_taken, sizeof(v)) != cudaSuccess) v = DeviceStatus{0u, 0u};
  return v;
}

}  // namespace sls
