// Arguments and page-list slicing shared by the attend kernels.
#pragma once

#include "common.cuh"

namespace sls {

struct AttendArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* page_idx;
  const int32_t* count;
  const int32_t* ctx_len;
  float* o_part;
  float* m_part;
  float* l_part;
  int idx_stride, k_fixed, S;
  int Hq, Hkv, G, Cap, P, pshift;
  float qscale;  // softmax scale * log2(e): scores are kept in base-2 units
};

// Slice [e0, e1) of row `row`'s page list handled by split `split`.
struct Slice {
  int N, e0, nent;
};
__device__ __forceinline__ Slice attend_slice(const AttendArgs& a, int row, int split) {
  const int b = row / a.Hkv;
  Slice sl;
  sl.N = clamp_len(a.ctx_len[b], a.Cap);
  int cnt;
  if (a.page_idx == nullptr) {
    cnt = (sl.N + a.P - 1) >> a.pshift;
  } else {
    cnt = a.count ? a.count[row] : a.k_fixed;
    cnt = cnt < 0 ? 0 : (cnt > a.idx_stride ? a.idx_stride : cnt);
  }
  const int per = (cnt + a.S - 1) / a.S;
  sl.e0 = split * per;
  const int e1 = min(sl.e0 + per, cnt);
  sl.nent = e1 > sl.e0 ? e1 - sl.e0 : 0;
  return sl;
}

// Position of a token given its page (or -1 when the slot is empty, the
// page is out of range or the position is past the context).
__device__ __forceinline__ int token_position(const AttendArgs& a, int pg, int j, int N) {
  if ((unsigned)pg >= (unsigned)(a.Cap >> a.pshift)) return -1;
  const int p = (pg << a.pshift) + (j & (a.P - 1));
  return p < N ? p : -1;
}

}  // namespace sls
