// Partial-tile visibility check shared by the kernels that traverse query rows (the forward and
// the dQ kernel): the unsigned interval test of CompileMask section 4.4.
#pragma once
#include <cmath>
#include <cstdint>

namespace cm {

// Replace invisible scores by -inf: key j0 + c is visible to the row iff for some interval
// (start, end): (u32)(j0 + c - start) < (u32)(end - start).
template <int NI, int N>
__device__ __forceinline__ void mask_cols(float (&s)[N], int j0, const int (&st)[4],
                                          const uint32_t (&len)[4]) {
  uint32_t base[NI];
#pragma unroll
  for (int n = 0; n < NI; ++n) base[n] = static_cast<uint32_t>(j0 - st[n]);
#pragma unroll
  for (int c = 0; c < N; ++c) {
    bool vis = false;
#pragma unroll
    for (int n = 0; n < NI; ++n) vis |= (base[n] + static_cast<uint32_t>(c)) < len[n];
    s[c] = vis ? s[c] : -INFINITY;
  }
}

}  // namespace cm
