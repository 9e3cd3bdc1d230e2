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

// Work item (index into the longest-first schedule) and head of CTA q of a grid of n_items * H
// CTAs.  Items are taken in chunks of kChunkItems in schedule order, and within a chunk the heads
// follow one another: the CTAs resident at one time then work on one or two (sample, head)s,
// whose K/V (or Q/dO) tiles stay in L2, while the longest rows of every head still start first.
constexpr int kChunkItems = 128;
__device__ __forceinline__ void cta_work(int q, int n_items, int H, int& item_idx, int& h) {
  const int full = n_items / kChunkItems;
  const int span = kChunkItems * H;
  if (q < full * span) {
    const int k = q / span, r = q - k * span;
    h = r / kChunkItems;
    item_idx = k * kChunkItems + (r - h * kChunkItems);
  } else {  // the last, partial chunk of rem items (rem > 0 here)
    const int r = q - full * span, rem = n_items - full * kChunkItems;
    h = r / rem;
    item_idx = full * kChunkItems + (r - h * rem);
  }
}

// Forms of the partial-tile visibility check (the ablation of CompileMask section 4.4):
//   kCheckUnsigned    visible iff (u32)(x - s) < (u32)(e - s) for some visible interval [s, e):
//                     one subtraction and one unsigned comparison per interval (the default);
//   kCheckTwoCompare  visible iff s <= x && x < e for some visible interval;
//   kCheckMasked      the complement of the visible intervals in [0, S) is used as a list of
//                     masked intervals (the FlashMask form), each tested with the unsigned
//                     comparison; visible iff x lies in none of them.
constexpr int kCheckUnsigned = 0;
constexpr int kCheckTwoCompare = 1;
constexpr int kCheckMasked = 2;

// One row's (or key column's) intervals in the form the check uses: start and length, and for
// the two-compare form the end.  The masked form holds up to NI + 1 gaps.
struct RowIntervals {
  int st[5];
  int en[5];
  uint32_t len[5];
};

// Loads the row's NI visible intervals from a slot-major Interval Table [b][NI][S][2]; for the
// masked form turns them into the gaps of their union within [0, S) (zero-length when unused).
__device__ __forceinline__ void load_row_intervals(const int32_t* itab, int b, int NI, int S, int row,
                                                   int check, RowIntervals& ri) {
  int s[4], e[4];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    s[n] = 0;
    e[n] = 0;
    if (n < NI) {
      const int2 iv = reinterpret_cast<const int2*>(itab)[(static_cast<size_t>(b) * NI + n) * S + row];
      s[n] = iv.x;
      e[n] = iv.y;
    }
  }
#pragma unroll
  for (int n = 0; n < 5; ++n) {
    ri.st[n] = n < 4 ? s[n] : 0;
    ri.en[n] = n < 4 ? e[n] : 0;
  }
  if (check == kCheckMasked) {
    // sort the non-empty intervals by start (empty ones last), then walk the gaps
#pragma unroll
    for (int n = 0; n < 4; ++n)
      if (e[n] <= s[n]) s[n] = 0x7FFFFFFF;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y + 1 < 4 - x; ++y)
        if (s[y] > s[y + 1]) {
          int u = s[y]; s[y] = s[y + 1]; s[y + 1] = u;
          u = e[y]; e[y] = e[y + 1]; e[y + 1] = u;
        }
    int cursor = 0;  // end of the visible union so far
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const bool live = s[n] != 0x7FFFFFFF;
      const int gs = cursor, ge = live ? (s[n] > cursor ? s[n] : cursor) : cursor;
      ri.st[n] = gs;
      ri.en[n] = ge;
      if (live && e[n] > cursor) cursor = e[n];
    }
    ri.st[4] = cursor;
    ri.en[4] = S;
  }
#pragma unroll
  for (int n = 0; n < 5; ++n) ri.len[n] = static_cast<uint32_t>(ri.en[n] - ri.st[n]);
}

// true iff x (= x0 + c) is visible under the given form; NI = the number of stored intervals
template <int NI, int CHECK>
__device__ __forceinline__ bool visible_at(uint32_t c, int x0, const RowIntervals& ri) {
  if (CHECK == kCheckMasked) {
    bool hidden = false;
#pragma unroll
    for (int n = 0; n < NI + 1; ++n) {
      const int k = n < NI ? n : 4;  // the gaps before each interval, then the tail gap
      hidden |= (static_cast<uint32_t>(x0 - ri.st[k]) + c) < ri.len[k];
    }
    return !hidden;
  }
  bool vis = false;
#pragma unroll
  for (int n = 0; n < NI; ++n) {
    if (CHECK == kCheckTwoCompare) {
      const int x = x0 + static_cast<int>(c);
      vis |= (x >= ri.st[n]) & (x < ri.en[n]);
    } else {
      vis |= (static_cast<uint32_t>(x0 - ri.st[n]) + c) < ri.len[n];
    }
  }
  return vis;
}

// Replace invisible scores by -inf: key j0 + c of the row (c < N).
template <int NI, int CHECK, int N>
__device__ __forceinline__ void mask_cols(float (&s)[N], int j0, const RowIntervals& ri) {
#pragma unroll
  for (int c = 0; c < N; ++c) s[c] = visible_at<NI, CHECK>(static_cast<uint32_t>(c), j0, ri) ? s[c] : -INFINITY;
}

// Bit c set iff index i0 + c (c < 32) is visible (the key-column form of the backward).
template <int NI, int CHECK>
__device__ __forceinline__ uint32_t visible_bits(int i0, const RowIntervals& ri) {
  uint32_t bits = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c) bits |= visible_at<NI, CHECK>(static_cast<uint32_t>(c), i0, ri) ? (1u << c) : 0u;
  return bits;
}

// Runtime dispatch over the interval count (1..4) and the check form.
template <int N>
__device__ __forceinline__ void mask_cols_any(float (&s)[N], int j0, const RowIntervals& ri, int NI,
                                              int check) {
#define CM_MASK_CASE(ni)                                                   \
  case ni:                                                                 \
    if (check == kCheckTwoCompare) mask_cols<ni, kCheckTwoCompare>(s, j0, ri); \
    else if (check == kCheckMasked) mask_cols<ni, kCheckMasked>(s, j0, ri);     \
    else mask_cols<ni, kCheckUnsigned>(s, j0, ri);                        \
    break;
  switch (NI) {
    CM_MASK_CASE(1)
    CM_MASK_CASE(2)
    CM_MASK_CASE(3)
    default:
      CM_MASK_CASE(4)
  }
#undef CM_MASK_CASE
}
__device__ __forceinline__ uint32_t visible_bits_any(int i0, const RowIntervals& ri, int NI, int check) {
#define CM_BITS_CASE(ni)                                                        \
  case ni:                                                                      \
    if (check == kCheckTwoCompare) return visible_bits<ni, kCheckTwoCompare>(i0, ri); \
    if (check == kCheckMasked) return visible_bits<ni, kCheckMasked>(i0, ri);         \
    return visible_bits<ni, kCheckUnsigned>(i0, ri);
  switch (NI) {
    CM_BITS_CASE(1)
    CM_BITS_CASE(2)
    CM_BITS_CASE(3)
    default:
      CM_BITS_CASE(4)
  }
#undef CM_BITS_CASE
}

}  // namespace cm
