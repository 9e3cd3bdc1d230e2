// Body of the online preprocess kernel for one direction of the Execution Descriptor
// (CompileMask sections 3.3 and 3.3.1).  It is shared by two kernels that differ only in the row
// evaluator, a template parameter:
//   - the generic kernel, which interprets the compiled endpoint programs, and
//   - the mask-specific kernels that the compiler generates from a MaskSpec and NVRTC builds at
//     run time (section 3.1: the compiler generates a mask-specific preprocess kernel).
//
// One block covers one 128-row tile of one sample; thread t owns row tile*128 + t:
//   1. the sample's segment boundaries are staged in shared memory and validated;
//   2. the evaluator gives each slot's raw endpoints; they are clamped to [0, S] and stored as
//      (start, end), with (0, 0) for padding, failed conditions and empty intervals; stores are
//      8-byte and coalesced (slot-major layout [b][slot][row]);
//   3. tile states: each row adds its touched tile ranges ("any") and the tile ranges its merged
//      intervals cover completely ("all") to two shared-memory difference arrays; a prefix sum
//      over the tiles gives, per tile, empty (no row touches it), full (all 128 rows cover it)
//      or partial.  A union of adjacent or overlapping slots counts as covering, so the states
//      equal those of the dense mask exactly;
//   4. the tile row's count of non-empty tiles goes to `rowcnt`, the input of the schedule.
//
// NVRTC compiles this header too, so it includes no standard-library header there.
#pragma once

#ifdef __CUDACC_RTC__
typedef int int32_t;
typedef unsigned int uint32_t;
typedef unsigned char uint8_t;
#else
#include <cstdint>
#endif

namespace cmcore {

constexpr int kTile = 128;
constexpr int kSlots = 4;          // most slots a row can have (the compiler's limit)
constexpr int kStatusBadMeta = 2;  // device status code: segment metadata failed validation

// Kernel parameters of one direction (forward: query rows; backward: key columns).
struct DescCore {
  int32_t* itab;        // [B][ni][S][2]
  uint32_t* bm;         // [B][NT][W]
  int32_t* rowcnt;      // [B][NT] non-empty tiles per tile row
  const int32_t* seg;   // [B][nseg_max + 1]
  const int32_t* nseg;  // [B]
  int32_t* status;      // device error word (first error wins)
  int nseg_max, B, S, NT, W, ni, dir;
};

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }
// wrapping int32 arithmetic: endpoint terms never overflow on valid metadata, and whatever they
// give on invalid metadata is clamped like any other value
__device__ __forceinline__ int wadd(int a, int b) {
  return static_cast<int>(static_cast<unsigned>(a) + static_cast<unsigned>(b));
}
__device__ __forceinline__ int wmul(int a, int c) {
  return static_cast<int>(static_cast<unsigned>(a) * static_cast<unsigned>(c));
}
// non-negative remainder by a positive constant
__device__ __forceinline__ int imod(int a, int c) {
  const int r = a % c;
  return r < 0 ? r + c : r;
}
// segment holding position e: the largest k in [0, nseg - 1] with seg[k] <= e
__device__ __forceinline__ int seg_index(const int* seg_s, int nseg, int e) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seg_s[mid] <= e) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ int seg_start_at(const int* seg_s, int nseg, int k) {
  return seg_s[imin(imax(k, 0), nseg)];
}
__device__ __forceinline__ int seg_end_at(const int* seg_s, int nseg, int k) {
  return seg_s[imin(imax(k, -1) + 1, nseg)];
}

// Adds v (+1 or -1; 0 for a lane with nothing to add) at index x of a shared-memory array.  The
// rows of one warp mostly update the same tile index, so a warp whose active lanes agree on x
// makes one atomic with their sum instead of up to 32 conflicting ones.  Call with the whole warp.
__device__ __forceinline__ void warp_add(int* arr, int x, int v) {
  const unsigned full = 0xFFFFFFFFu;
  const int lo = __reduce_min_sync(full, v != 0 ? x : 0x7FFFFFFF);
  const int hi = __reduce_max_sync(full, v != 0 ? x : -1);
  if (lo == hi) {
    const int sum = __reduce_add_sync(full, v);
    if ((threadIdx.x & 31) == 0 && sum != 0) atomicAdd(&arr[lo], sum);
  } else if (lo < hi && v != 0) {
    atomicAdd(&arr[x], v);
  }
}

// Dynamic shared memory: (nseg_max + 1) + 2 * (NT + 1) ints + NT bytes.
// NS: the slots the evaluator may fill, known at compile time; slots n >= p.ni are not stored.
// Eval::row(i, seg_idx(i), seg, nseg, S, lo, hi) writes raw endpoints of the row's slots and
// leaves lo = hi = 0 in slots the row does not have.
template <int NS, class Eval>
__device__ __forceinline__ void descriptor_tile(const DescCore& p, int b, int tile, const Eval& ev) {
  extern __shared__ int smem_i[];
  __shared__ int s_bad;
  __shared__ int s_wtot[3][kTile / 32];
  int* seg_s = smem_i;                     // [nseg_max + 1]
  int* cnt_any = smem_i + p.nseg_max + 1;  // [NT + 1] difference array: rows touching a tile
  int* cnt_all = cnt_any + p.NT + 1;       // [NT + 1] difference array: rows covering a tile
  uint8_t* code = reinterpret_cast<uint8_t*>(cnt_all + p.NT + 1);  // [NT] 2-bit state per tile

  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  int nseg = p.nseg[b];
  if (t == 0) s_bad = (nseg < 1 || nseg > p.nseg_max);
  nseg = imin(imax(nseg, 1), p.nseg_max);
  for (int k = t; k <= p.nseg_max; k += blockDim.x) seg_s[k] = p.seg[b * (p.nseg_max + 1) + k];
  for (int k = t; k < 2 * (p.NT + 1); k += blockDim.x) cnt_any[k] = 0;
  __syncthreads();
  // metadata validation: seg[0] = 0, strictly increasing, seg[nseg] = S
  bool bad = false;
  for (int k = t; k < nseg; k += blockDim.x) bad |= seg_s[k + 1] <= seg_s[k];
  if (t == 0) bad |= seg_s[0] != 0 || seg_s[nseg] != p.S;
  if (bad) s_bad = 1;
  __syncthreads();
  if (s_bad && t == 0 && tile == 0 && p.status != nullptr)
    atomicCAS(p.status, 0, (kStatusBadMeta << 16) | p.dir);

  // --- 1. endpoints ---------------------------------------------------------------------------
  const int row = tile * kTile + t;
  int lo[NS], hi[NS];
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    lo[n] = 0;
    hi[n] = 0;
  }
  ev.row(row, seg_index(seg_s, nseg, row), seg_s, nseg, p.S, lo, hi);
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    int a = imin(imax(lo[n], 0), p.S);
    int e = imin(imax(hi[n], 0), p.S);
    if (n >= p.ni || e <= a) {
      a = 0;
      e = 0;
    }
    lo[n] = a;
    hi[n] = e;
    if (n < p.ni) {
      int2* dst = reinterpret_cast<int2*>(p.itab) +
                  (static_cast<unsigned long long>(b) * p.ni + n) * p.S + row;
      *dst = make_int2(a, e);
    }
  }

  // --- 2. merged intervals (sorted by start; overlapping or adjacent ones joined) -------------
  int ms[NS], me[NS];
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    ms[n] = hi[n] > lo[n] ? lo[n] : 0x7FFFFFFF;
    me[n] = hi[n];
  }
#pragma unroll
  for (int x = 0; x < NS; ++x)
#pragma unroll
    for (int y = 0; y + 1 < NS - x; ++y)
      if (ms[y] > ms[y + 1]) {
        int u = ms[y]; ms[y] = ms[y + 1]; ms[y + 1] = u;
        u = me[y]; me[y] = me[y + 1]; me[y + 1] = u;
      }
#pragma unroll
  for (int n = 1; n < NS; ++n) {
    if (ms[n] != 0x7FFFFFFF && ms[n] <= me[n - 1] && ms[n - 1] != 0x7FFFFFFF) {
      ms[n] = ms[n - 1];
      me[n] = imax(me[n], me[n - 1]);
      ms[n - 1] = 0x7FFFFFFF;  // absorbed
    }
  }

  // --- 3. tile states ---------------------------------------------------------------------------
  // +1 / -1 at the ends of the row's touched tile ranges (any slot) and of its fully covered tile
  // ranges (merged intervals, disjoint, so a row counts once per tile).  After the prefix sum a
  // tile is touched iff its "any" count is > 0 and full iff its "all" count is 128.
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    const bool touch = hi[n] > lo[n];
    warp_add(cnt_any, lo[n] / kTile, touch ? 1 : 0);
    warp_add(cnt_any, touch ? (hi[n] - 1) / kTile + 1 : 0, touch ? -1 : 0);
    const bool merged = ms[n] != 0x7FFFFFFF;
    const int a = merged ? (ms[n] + kTile - 1) / kTile : 0;
    const int e = merged ? me[n] / kTile : 0;
    const bool cover = merged && e > a;
    warp_add(cnt_all, a, cover ? 1 : 0);
    warp_add(cnt_all, e, cover ? -1 : 0);
  }
  __syncthreads();
  // block prefix sum: thread t owns tiles [t * per, (t + 1) * per)
  const int per = (p.NT + kTile - 1) / kTile;
  const int c0 = t * per;
  int sa = 0, sf = 0;
  for (int c = c0; c < c0 + per && c < p.NT; ++c) {
    sa += cnt_any[c];
    sf += cnt_all[c];
  }
  int ia = sa, iff = sf;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xFFFFFFFFu, ia, o);
    const int yf = __shfl_up_sync(0xFFFFFFFFu, iff, o);
    if (lane >= o) {
      ia += ya;
      iff += yf;
    }
  }
  if (lane == 31) {
    s_wtot[0][warp] = ia;
    s_wtot[1][warp] = iff;
  }
  __syncthreads();
  int run_a = ia - sa, run_f = iff - sf;  // exclusive prefix within the warp
  for (int w = 0; w < warp; ++w) {
    run_a += s_wtot[0][w];
    run_f += s_wtot[1][w];
  }
  int nonempty = 0;
  for (int c = c0; c < c0 + per && c < p.NT; ++c) {
    run_a += cnt_any[c];
    run_f += cnt_all[c];
    code[c] = run_a > 0 ? (run_f == kTile ? 2 : 1) : 0;
    nonempty += run_a > 0 ? 1 : 0;
  }
  nonempty = __reduce_add_sync(0xFFFFFFFFu, nonempty);
  if (lane == 0) s_wtot[2][warp] = nonempty;
  __syncthreads();
  if (t == 0) {
    int total = 0;
#pragma unroll
    for (int w = 0; w < kTile / 32; ++w) total += s_wtot[2][w];
    p.rowcnt[static_cast<unsigned long long>(b) * p.NT + tile] = total;
  }
  uint32_t* out = p.bm + (static_cast<unsigned long long>(b) * p.NT + tile) * p.W;
  for (int ow = t; ow < p.W; ow += blockDim.x) {
    uint32_t word = 0;
    for (int q = 0; q < 16; ++q) {
      const int c = ow * 16 + q;
      if (c >= p.NT) break;
      word |= static_cast<uint32_t>(code[c]) << (2 * q);
    }
    out[ow] = word;
  }
}

}  // namespace cmcore
