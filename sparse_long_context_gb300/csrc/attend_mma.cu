// Tensor-core attend kernel (bf16).  Not built yet: every call falls back to
// the CUDA-core kernel in attend.cu.
#include "attend_common.cuh"
#include "launch.h"

namespace sls {

cudaError_t launch_attend_mma(const Shape&, const AttendArgs&, cudaStream_t, bool* handled) {
  *handled = false;
  return cudaSuccess;
}

}  // namespace sls
