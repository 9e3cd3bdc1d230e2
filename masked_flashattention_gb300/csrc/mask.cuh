// Helpers shared by the attention kernels: walking the non-empty tiles of a Tile-State Bitmap row
// (CompileMask section 3.3.1) and the partial-tile visibility check (section 3.3.2; the unsigned
// interval test of section 4.4 and the other forms of its ablation).
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

// Work queue of a persistent attention kernel (two ints in the descriptor's work buffer): q[0]
// hands out work items in schedule order to whichever CTA asks next, q[1] counts the CTAs that
// have finished.  The last CTA of a launch returns both to zero, ready for the next launch (every
// CTA has taken its last item before it counts itself finished).
__device__ __forceinline__ void queue_finish(int* q) {
  __threadfence();
  if (atomicAdd(q + 1, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(q, 0);
    atomicExch(q + 1, 0);
    __threadfence();
  }
}

// Forms of the partial-tile visibility check (full and empty tiles never run one):
//   kCheckUnsigned    per score: for each stored interval [s, e) one subtraction and one unsigned
//                     comparison, (u32)(x - s) < (u32)(e - s) (the paper's section 4.4 test);
//   kCheckTwoCompare  per score: s <= x && x < e for each stored interval;
//   kCheckRangeMask   per row and 32-index chunk [x0, x0 + 32): each stored interval becomes the
//                     bit range [clamp(s - x0), clamp(e - x0)) of a 32-bit mask (two clamped
//                     subtractions and two funnel shifts), and each score then tests one bit
//                     (the default: the per-score cost no longer grows with the interval count).
// The stored intervals are the row's visible intervals (visible form of the descriptor) or the
// masked intervals of their complement in [0, S) (masked form, the representation the pages
// compare against in section 4.4): in the masked form an index is visible iff it lies in none.
constexpr int kCheckUnsigned = 0;
constexpr int kCheckTwoCompare = 1;
constexpr int kCheckRangeMask = 3;

constexpr int kMaxStored = 9;  // up to 8 visible intervals, or the 9 gaps around them

// A row's stored intervals in registers.  The kernels are compiled for two capacities, MAXNI = 4
// (every workload here in the visible form) and 9, so that the common case keeps few registers.
template <int MAXNI>
struct RowIntervals {
  int st[MAXNI];
  int en[MAXNI];
};

// Loads the row's NI stored intervals from a slot-major Interval Table [b][NI][S][2] (unused
// registers hold the empty interval (0, 0)).
template <int MAXNI>
__device__ __forceinline__ void load_row_intervals(const int32_t* itab, int b, int NI, int S,
                                                   int row, RowIntervals<MAXNI>& ri) {
#pragma unroll
  for (int n = 0; n < MAXNI; ++n) {
    ri.st[n] = 0;
    ri.en[n] = 0;
    if (n < NI) {
      const int2 iv = reinterpret_cast<const int2*>(itab)[(static_cast<size_t>(b) * NI + n) * S + row];
      ri.st[n] = iv.x;
      ri.en[n] = iv.y;
    }
  }
}

// ---- per-score forms ----------------------------------------------------------------------------
// true iff x0 + c lies in one of the first NI stored intervals
template <int NI, int CHECK, class RI>
__device__ __forceinline__ bool in_any(uint32_t c, int x0, const RI& ri) {
  bool in = false;
#pragma unroll
  for (int n = 0; n < NI; ++n) {
    if (CHECK == kCheckTwoCompare) {
      const int x = x0 + static_cast<int>(c);
      in |= (x >= ri.st[n]) & (x < ri.en[n]);
    } else {
      in |= (static_cast<uint32_t>(x0 - ri.st[n]) + c) <
            static_cast<uint32_t>(ri.en[n] - ri.st[n]);
    }
  }
  return in;
}

// Replace invisible scores by -inf: key j0 + c of the row (c < N).
template <int NI, int CHECK, int N, class RI>
__device__ __forceinline__ void mask_cols(float (&s)[N], int j0, const RI& ri, bool masked) {
#pragma unroll
  for (int c = 0; c < N; ++c)
    s[c] = (in_any<NI, CHECK>(static_cast<uint32_t>(c), j0, ri) != masked) ? s[c] : -INFINITY;
}

// Bit c set iff index i0 + c (c < 32) is visible.
template <int NI, int CHECK, class RI>
__device__ __forceinline__ uint32_t visible_bits(int i0, const RI& ri, bool masked) {
  uint32_t bits = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c)
    bits |= (in_any<NI, CHECK>(static_cast<uint32_t>(c), i0, ri) != masked) ? (1u << c) : 0u;
  return bits;
}

// ---- range-mask form -----------------------------------------------------------------------------
// Bits [clamp(s - x0, 0, 32), clamp(e - x0, 0, 32)) of a 32-bit word: the indices of the chunk
// [x0, x0 + 32) inside [s, e).  The funnel shift of 0xFFFFFFFF by n (clamped at 32) into a zero
// high word gives the n lowest bits set.
__device__ __forceinline__ uint32_t low_bits(int n) {
  return __funnelshift_lc(0xFFFFFFFFu, 0u, static_cast<uint32_t>(n > 0 ? n : 0));
}
template <int MAXNI>
__device__ __forceinline__ uint32_t range_bits(const RowIntervals<MAXNI>& ri, int NI, int x0,
                                               bool masked) {
  uint32_t m = 0;
#pragma unroll
  for (int n = 0; n < MAXNI; ++n)
    if (n < NI) m |= low_bits(ri.en[n] - x0) & ~low_bits(ri.st[n] - x0);
  return masked ? ~m : m;
}

// Scores of 32 keys [j0, j0 + 32) whose bit in `vis` is clear become -inf.  The warp skips the
// chunk when every lane's mask is full.
__device__ __forceinline__ void apply_bits(float* s, uint32_t vis) {
  if (__all_sync(0xFFFFFFFFu, vis == 0xFFFFFFFFu)) return;
#pragma unroll
  for (int c = 0; c < 32; ++c) s[c] = (vis & (1u << c)) ? s[c] : -INFINITY;
}

// ---- dispatch ------------------------------------------------------------------------------------
// Masks N (a multiple of 32) scores of keys [j0, j0 + N) of one row: NI stored intervals (1..9),
// `check` one of the forms above, `masked` the descriptor form.
template <int N, int MAXNI>
__device__ __forceinline__ void mask_cols_any(float (&s)[N], int j0, const RowIntervals<MAXNI>& ri,
                                              int NI, int check, bool masked) {
  if (check == kCheckRangeMask) {
#pragma unroll
    for (int q = 0; q < N / 32; ++q) apply_bits(&s[32 * q], range_bits(ri, NI, j0 + 32 * q, masked));
    return;
  }
#define CM_MASK_CASE(ni)                                                                  \
  case ni:                                                                                \
    if constexpr (ni <= MAXNI) {                                                          \
      if (check == kCheckTwoCompare) mask_cols<ni, kCheckTwoCompare>(s, j0, ri, masked);   \
      else mask_cols<ni, kCheckUnsigned>(s, j0, ri, masked);                              \
    }                                                                                     \
    break;
  switch (NI) {
    CM_MASK_CASE(1)
    CM_MASK_CASE(2)
    CM_MASK_CASE(3)
    CM_MASK_CASE(4)
    CM_MASK_CASE(5)
    CM_MASK_CASE(6)
    CM_MASK_CASE(7)
    CM_MASK_CASE(8)
    CM_MASK_CASE(9)
    default:
      break;
  }
#undef CM_MASK_CASE
}

// Visibility bits of the 32 indices [i0, i0 + 32) (the key-column form of the backward).
template <int MAXNI>
__device__ __forceinline__ uint32_t visible_bits_any(int i0, const RowIntervals<MAXNI>& ri, int NI,
                                                     int check, bool masked) {
  if (check == kCheckRangeMask) return range_bits(ri, NI, i0, masked);
#define CM_BITS_CASE(ni)                                                                     \
  case ni:                                                                                   \
    if constexpr (ni <= MAXNI) {                                                             \
      if (check == kCheckTwoCompare) return visible_bits<ni, kCheckTwoCompare>(i0, ri, masked); \
      return visible_bits<ni, kCheckUnsigned>(i0, ri, masked);                               \
    }                                                                                        \
    break;
  switch (NI) {
    CM_BITS_CASE(1)
    CM_BITS_CASE(2)
    CM_BITS_CASE(3)
    CM_BITS_CASE(4)
    CM_BITS_CASE(5)
    CM_BITS_CASE(6)
    CM_BITS_CASE(7)
    CM_BITS_CASE(8)
    CM_BITS_CASE(9)
    default:
      break;
  }
  return 0u;
#undef CM_BITS_CASE
}

}  // namespace cm
