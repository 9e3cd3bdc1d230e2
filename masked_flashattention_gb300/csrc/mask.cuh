// Helpers shared by the attention kernels: walking the non-empty tiles of a Tile-State Bitmap row
// (CompileMask section 3.3.1) and the partial-tile visibility check of the kernels that traverse
// query rows (the unsigned interval test of section 4.4).
#pragma once
#include <cmath>
#include <cstdint>

namespace cm {

// first tile c' >= c whose 2-bit state in the bitmap row is not empty, or NT
__device__ __forceinline__ int next_tile(const uint32_t* row, int NT, int c) {
  while (c < NT) {
    const int w = c >> 4;
    uint32_t x = row[w];
    x = (x | (x >> 1)) & 0x55555555u;
    x &= 0xFFFFFFFFu << (2 * (c & 15));
    if (x != 0) return (w << 4) + ((__ffs(x) - 1) >> 1);
    c = (w + 1) << 4;
  }
  return NT;
}
__device__ __forceinline__ bool tile_is_full(const uint32_t* row, int c) {
  return ((row[c >> 4] >> (2 * (c & 15))) & 3u) == 2u;
}

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
