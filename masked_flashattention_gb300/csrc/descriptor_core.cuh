// Body of the online preprocess kernel (CompileMask sections 3.3 and 3.3.1): one launch builds
// both halves of the Execution Descriptor (forward: query rows; backward: key columns) and their
// longest-first schedules.  It is shared by two kernels that differ only in their row evaluators
// (template parameters):
//   - the generic kernel, which interprets the compiled endpoint programs, and
//   - the mask-specific kernels that the compiler generates from a pair of MaskSpecs and NVRTC
//     builds at run time (section 3.1: the compiler generates a mask-specific preprocess kernel).
//
// Work is split into units of 4 tile rows (4 x 128 rows) of one (direction, sample); a block of
// 4 warps takes a contiguous range of units (the grid is sized to be resident at once and
// launched cooperatively).  Warp w of a unit owns one tile row, lane l its rows 4l .. 4l + 3:
//   1. the sample's segment boundaries are staged in shared memory and validated;
//   2. the evaluator gives each slot's raw endpoints per row; they are clamped to [0, S] and kept
//      as (start, end), with (0, 0) for padding, failed conditions and empty intervals.  The
//      visible form stores them as they are, the masked form the maximal runs of invisible
//      indices; either way a lane writes each slot's 4 rows with two 16-byte stores (slot-major
//      layout [b][slot][row], so a warp's stores cover 1 KB contiguously);
//   3. tile states: each row's touched tile ranges (any slot) and fully covered tile ranges
//      (merged intervals) go into one shared-memory difference array per warp, touched counts in
//      the low 16 bits and covered counts in the high 16 bits.  Lanes whose 4 rows agree and share
//      a range with other lanes add it once for all of them.  A prefix sum over the tiles gives,
//      per tile, empty (no row touches it), full (all 128 rows cover it) or partial.  A union of
//      adjacent or overlapping slots counts as covering, so the states equal the dense mask's;
//   4. the tile row's count of non-empty tiles takes a ticket in a global histogram per
//      direction.  After a grid barrier every block reads the histogram, and each tile row is
//      placed at (rows with more tiles) + ticket: a counting sort, longest first, ties in any
//      order.
//
// NVRTC compiles this header too, so it includes no standard-library header there.
#pragma once

#ifdef __CUDACC_RTC__
typedef int int32_t;
typedef unsigned int uint32_t;
typedef unsigned char uint8_t;
typedef unsigned long long uint64_t;
#else
#include <cstdint>
#endif

namespace cmcore {

constexpr int kTile = 128;
constexpr int kSlots = 8;          // most slots a row can have (the compiler's limit)
constexpr int kWarps = 4;          // tile rows per work unit, warps per block
constexpr int kThreads = 32 * kWarps;
constexpr int kRowsPerLane = kTile / 32;
constexpr int kStatusTimeout = 1;  // device status codes (first error wins)
constexpr int kStatusBadMeta = 2;
constexpr int kNone = 0x7FFFFFFF;

// One half of the descriptor.
struct DescDir {
  int32_t* itab;   // [B][ni][S][2]
  uint32_t* bm;    // [B][NT][W]
  int32_t* sched;  // [B * NT]
  int ni;          // stored slots per row: the spec's slots (visible form) or one more (masked)
};

// Kernel parameters.
struct DescCore {
  DescDir dir[2];        // 0 forward, 1 backward
  const int32_t* seg;    // [B][nseg_max + 1]
  const int32_t* nseg;   // [B]
  int32_t* work;         // zeroed before the launch: [0] status word, [1] grid barrier count,
                         // [2 + d * (NT + 1) + c] tile rows of direction d with c non-empty tiles
  int nseg_max, B, S, NT, W;
  int groups;            // work units per (direction, sample): ceil(NT / kWarps)
  int units_per_block;   // most units a block takes (sizes its list of tile rows)
  int masked;            // 1: store the masked runs instead of the visible intervals
  uint64_t wait_ns;      // limit of the grid barrier wait
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

__device__ __forceinline__ void record_status(int32_t* work, int code, int where) {
  atomicCAS(work, 0, (code << 16) | (where & 0xFFFF));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Every block of the (cooperative, fully resident) grid arrives, then waits until all have.  The
// wait is bounded: past wait_ns it records a time-out and returns.
__device__ __forceinline__ void grid_barrier(const DescCore& p) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&p.work[1], 1);
    const int n = static_cast<int>(gridDim.x);
    if (ld_acquire(&p.work[1]) < n) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(&p.work[1]) < n) {
        if (globaltimer_ns() - t0 > p.wait_ns) {
          record_status(p.work, kStatusTimeout, 0x400);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// Index of tile entry t in a warp's difference array: one padding word per 32 entries, so that the
// prefix pass (lane l walks entries [l * per, (l + 1) * per)) reads 32 different banks.
__device__ __forceinline__ int cidx(int t) { return t + (t >> 5); }

// Adds `unit` rows over the tile range [key >> 16, key & 0xFFFF) of the warp's difference array
// for each of the lane's 4 rows (key 0xFFFFFFFF: no range).  When the 4 rows agree, lanes with
// the same range are added together by one leader.  Call with the whole warp.
__device__ __forceinline__ void add_ranges(int* cnt, const uint32_t (&key)[kRowsPerLane], int unit) {
  const bool same = key[1] == key[0] && key[2] == key[0] && key[3] == key[0];
  const uint32_t k0 = same ? key[0] : 0xFFFFFFFEu;
  const unsigned grp = __match_any_sync(0xFFFFFFFFu, k0);
  const int lane = threadIdx.x & 31;
  if (same) {
    if (k0 != 0xFFFFFFFFu && lane == __ffs(grp) - 1) {
      const int w = kRowsPerLane * __popc(grp) * unit;
      atomicAdd(&cnt[cidx(k0 >> 16)], w);
      atomicAdd(&cnt[cidx(k0 & 0xFFFF)], -w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kRowsPerLane; ++q)
      if (key[q] != 0xFFFFFFFFu) {
        atomicAdd(&cnt[cidx(key[q] >> 16)], unit);
        atomicAdd(&cnt[cidx(key[q] & 0xFFFF)], -unit);
      }
  }
}

// One tile row of one direction: Interval Table rows, bitmap row; returns the number of non-empty
// tiles (in every lane).  NS: the slots the evaluator may fill, known at compile time; slots
// n >= ni - masked are not part of the spec.  Eval::row(i, seg_idx(i), seg, nseg, S, lo, hi)
// writes raw endpoints of the row's slots and leaves lo = hi = 0 in slots the row does not have.
template <int NS, class Eval>
__device__ __forceinline__ int tile_row(const DescCore& p, const DescDir& dd, int b, int tile,
                                        const int* seg_s, int nseg, int* cnt, const Eval& ev) {
  const int lane = threadIdx.x & 31;
  const int r0 = tile * kTile + lane * kRowsPerLane;
  const int spec_slots = dd.ni - p.masked;
  int lo[kRowsPerLane][NS], hi[kRowsPerLane][NS];

  // --- 1. endpoints: segment of the first row by binary search, then one step at most per row
  int k = seg_index(seg_s, nseg, r0);
#pragma unroll
  for (int q = 0; q < kRowsPerLane; ++q) {
    const int i = r0 + q;
    if (q > 0 && k + 1 < nseg && seg_s[k + 1] <= i) ++k;
#pragma unroll
    for (int n = 0; n < NS; ++n) {
      lo[q][n] = 0;
      hi[q][n] = 0;
    }
    ev.row(i, k, seg_s, nseg, p.S, lo[q], hi[q]);
#pragma unroll
    for (int n = 0; n < NS; ++n) {
      const int a = imin(imax(lo[q][n], 0), p.S);
      const int e = imin(imax(hi[q][n], 0), p.S);
      const bool keep = n < spec_slots && e > a;
      lo[q][n] = keep ? a : 0;
      hi[q][n] = keep ? e : 0;
    }
  }
  if (!p.masked) {
#pragma unroll
    for (int n = 0; n < NS; ++n) {
      if (n < dd.ni) {
        int4* dst = reinterpret_cast<int4*>(
            dd.itab + ((static_cast<unsigned long long>(b) * dd.ni + n) * p.S + r0) * 2);
        dst[0] = make_int4(lo[0][n], hi[0][n], lo[1][n], hi[1][n]);
        dst[1] = make_int4(lo[2][n], hi[2][n], lo[3][n], hi[3][n]);
      }
    }
  }

  // --- 2. merged intervals per row (sorted by start; overlapping or adjacent ones joined) -----
  int ms[kRowsPerLane][NS], me[kRowsPerLane][NS];
#pragma unroll
  for (int q = 0; q < kRowsPerLane; ++q) {
#pragma unroll
    for (int n = 0; n < NS; ++n) {
      ms[q][n] = hi[q][n] > lo[q][n] ? lo[q][n] : kNone;
      me[q][n] = hi[q][n];
    }
#pragma unroll
    for (int x = 0; x < NS; ++x)
#pragma unroll
      for (int y = 0; y + 1 < NS - x; ++y)
        if (ms[q][y] > ms[q][y + 1]) {
          int u = ms[q][y]; ms[q][y] = ms[q][y + 1]; ms[q][y + 1] = u;
          u = me[q][y]; me[q][y] = me[q][y + 1]; me[q][y + 1] = u;
        }
#pragma unroll
    for (int n = 1; n < NS; ++n) {
      if (ms[q][n] != kNone && ms[q][n - 1] != kNone && ms[q][n] <= me[q][n - 1]) {
        ms[q][n] = ms[q][n - 1];
        me[q][n] = imax(me[q][n], me[q][n - 1]);
        ms[q][n - 1] = kNone;  // absorbed
      }
    }
  }

  if (p.masked) {
    // Masked form: the gaps of the merged intervals in [0, S), in increasing order, then (0, 0)
    // padding (at most NS + 1 runs).
    int gs[kRowsPerLane][NS + 1], ge[kRowsPerLane][NS + 1];
#pragma unroll
    for (int q = 0; q < kRowsPerLane; ++q) {
      int cursor = 0;
#pragma unroll
      for (int n = 0; n < NS; ++n) {
        const bool live = ms[q][n] != kNone;
        gs[q][n] = live && ms[q][n] > cursor ? cursor : kNone;
        ge[q][n] = live ? ms[q][n] : 0;
        if (live) cursor = me[q][n];
      }
      gs[q][NS] = cursor < p.S ? cursor : kNone;
      ge[q][NS] = p.S;
      // the non-empty runs are already increasing: move the empty ones behind them
#pragma unroll
      for (int x = 0; x < NS + 1; ++x)
#pragma unroll
        for (int y = 0; y + 1 < NS + 1 - x; ++y)
          if (gs[q][y] > gs[q][y + 1]) {
            int u = gs[q][y]; gs[q][y] = gs[q][y + 1]; gs[q][y + 1] = u;
            u = ge[q][y]; ge[q][y] = ge[q][y + 1]; ge[q][y + 1] = u;
          }
#pragma unroll
      for (int n = 0; n < NS + 1; ++n)
        if (gs[q][n] == kNone) {
          gs[q][n] = 0;
          ge[q][n] = 0;
        }
    }
#pragma unroll
    for (int n = 0; n < NS + 1; ++n) {
      if (n < dd.ni) {
        int4* dst = reinterpret_cast<int4*>(
            dd.itab + ((static_cast<unsigned long long>(b) * dd.ni + n) * p.S + r0) * 2);
        dst[0] = make_int4(gs[0][n], ge[0][n], gs[1][n], ge[1][n]);
        dst[1] = make_int4(gs[2][n], ge[2][n], gs[3][n], ge[3][n]);
      }
    }
  }

  // --- 3. tile states ---------------------------------------------------------------------------
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    uint32_t touch[kRowsPerLane], cover[kRowsPerLane];
#pragma unroll
    for (int q = 0; q < kRowsPerLane; ++q) {
      // tiles [lo / 128, (hi - 1) / 128] touched by slot n
      touch[q] = hi[q][n] > lo[q][n]
                     ? (static_cast<uint32_t>(lo[q][n] >> 7) << 16) |
                           static_cast<uint32_t>(((hi[q][n] - 1) >> 7) + 1)
                     : 0xFFFFFFFFu;
      // tiles [ceil(ms / 128), me / 128) covered by merged interval n
      const int a = (ms[q][n] + kTile - 1) >> 7, e = me[q][n] >> 7;
      cover[q] = ms[q][n] != kNone && e > a
                     ? (static_cast<uint32_t>(a) << 16) | static_cast<uint32_t>(e)
                     : 0xFFFFFFFFu;
    }
    add_ranges(cnt, touch, 1);
    add_ranges(cnt, cover, 1 << 16);
  }
  __syncwarp();
  // prefix sum over the tiles: lane l owns tiles [l * per, (l + 1) * per), per a power of two;
  // entries are cleared as they are read, so the array is zero again for the next tile row
  int per = 1;
  while (per * 32 < p.NT) per <<= 1;
  const int t0 = lane * per;
  int run = 0;
#pragma unroll 4
  for (int q = 0; q < per; ++q)
    if (t0 + q < p.NT) run += cnt[cidx(t0 + q)];
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  int acc = incl - run;
  int nonempty = 0;
  uint32_t frag_lo = 0, frag_hi = 0;  // 2-bit codes of this lane's tiles
#pragma unroll 4
  for (int q = 0; q < per; ++q) {
    const int t = t0 + q;
    if (t < p.NT) {
      acc += cnt[cidx(t)];
      cnt[cidx(t)] = 0;
      const int touched = acc & 0xFFFF;
      const int covered = static_cast<int>(static_cast<uint32_t>(acc) >> 16);
      const uint32_t c = touched > 0 ? (covered == kTile ? 2u : 1u) : 0u;
      if (q < 16) frag_lo |= c << (2 * q);
      else frag_hi |= c << (2 * (q - 16));
      nonempty += touched > 0 ? 1 : 0;
    }
  }
  if (lane == 0) cnt[cidx(p.NT)] = 0;
  nonempty = __reduce_add_sync(0xFFFFFFFFu, nonempty);
  // bitmap words: 16 tiles each, from the lanes' code fragments
  uint32_t* out = dd.bm + (static_cast<unsigned long long>(b) * p.NT + tile) * p.W;
  if (per >= 16) {
    const int w0 = t0 >> 4;
    if (w0 < p.W) out[w0] = frag_lo;
    if (per == 32 && w0 + 1 < p.W) out[w0 + 1] = frag_hi;
  } else {
    const int lanes = 16 / per;  // lanes per word (a power of two)
    uint32_t word = frag_lo << (2 * per * (lane & (lanes - 1)));
    for (int o = 1; o < lanes; o <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, o);
    const int w = lane / lanes;
    if ((lane & (lanes - 1)) == 0 && w < p.W) out[w] = word;
  }
  __syncwarp();
  return nonempty;
}

// Dynamic shared memory of the kernel, in ints.
__host__ __device__ __forceinline__ int seg_ints(int nseg_max) { return (nseg_max + 1 + 3) & ~3; }
__host__ __device__ __forceinline__ int cnt_ints(int NT) { return (NT + 1 + (NT >> 5) + 3) & ~3; }
__host__ __device__ __forceinline__ int smem_ints(int nseg_max, int NT, int units_per_block) {
  return seg_ints(nseg_max) + kWarps * cnt_ints(NT) + 2 * kWarps * units_per_block;
}

template <int NSF, int NSB, class EvalF, class EvalB>
__device__ __forceinline__ void descriptor_kernel(const DescCore& p, const EvalF& evf,
                                                  const EvalB& evb) {
  extern __shared__ int smem_i[];
  __shared__ int s_bad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* seg_s = smem_i;
  int* cnt_all = seg_s + seg_ints(p.nseg_max);
  int* cnt = cnt_all + warp * cnt_ints(p.NT);
  int2* items = reinterpret_cast<int2*>(cnt_all + kWarps * cnt_ints(p.NT));
  int* hist = p.work + 2;

  for (int t = lane; t < cnt_ints(p.NT); t += 32) cnt[t] = 0;

  // ---- phase 1: tile rows ---------------------------------------------------------------------
  // block x takes the contiguous units [x * units_per_block, ...): consecutive units mostly share
  // a sample, so its segment boundaries are staged once for many tile rows
  const int per_dir = p.B * p.groups;
  const int u_begin = blockIdx.x * p.units_per_block;
  const int u_end = imin(u_begin + p.units_per_block, 2 * per_dir);
  int cur_b = -1, nseg = 1, u = 0;
  for (int unit = u_begin; unit < u_end; ++unit, ++u) {
    const int d = unit >= per_dir ? 1 : 0;
    const int rem = unit - d * per_dir;
    const int b = rem / p.groups, g = rem - b * p.groups;
    if (b != cur_b) {
      __syncthreads();  // no warp reads the previous sample's boundaries any more
      const int ns = p.nseg[b];
      nseg = imin(imax(ns, 1), p.nseg_max);
      if (threadIdx.x == 0) s_bad = ns < 1 || ns > p.nseg_max;
      for (int k = threadIdx.x; k <= p.nseg_max; k += kThreads)
        seg_s[k] = p.seg[b * (p.nseg_max + 1) + k];
      __syncthreads();
      // metadata validation: seg[0] = 0, strictly increasing, seg[nseg] = S
      bool bad = false;
      for (int k = threadIdx.x; k < nseg; k += kThreads) bad |= seg_s[k + 1] <= seg_s[k];
      if (threadIdx.x == 0) bad |= seg_s[0] != 0 || seg_s[nseg] != p.S;
      if (bad) s_bad = 1;
      __syncthreads();
      if (s_bad && threadIdx.x == 0) record_status(p.work, kStatusBadMeta, d);
      cur_b = b;
    }
    const int tile = g * kWarps + warp;
    int2 it = make_int2(-1, 0);
    if (tile < p.NT) {
      const int c = d == 0 ? tile_row<NSF>(p, p.dir[0], b, tile, seg_s, nseg, cnt, evf)
                           : tile_row<NSB>(p, p.dir[1], b, tile, seg_s, nseg, cnt, evb);
      it = make_int2(static_cast<int>((static_cast<uint32_t>(d) << 31) |
                                      (static_cast<uint32_t>(b) << 16) | static_cast<uint32_t>(tile)),
                     c);
    }
    if (lane == 0) items[u * kWarps + warp] = it;
  }
  const int n_items = u * kWarps;
  // tickets in the per-direction histograms, taken together so that their latencies overlap
  __syncthreads();
  for (int x = threadIdx.x; x < n_items; x += kThreads) {
    const int2 it = items[x];
    if (it.x == -1) continue;
    const int d = static_cast<int>(static_cast<uint32_t>(it.x) >> 31);
    const int ticket = atomicAdd(&hist[d * (p.NT + 1) + it.y], 1);
    items[x].y = (it.y << 16) | ticket;
  }

  // ---- phase 2: schedules ----------------------------------------------------------------------
  grid_barrier(p);
  // first position of each count: base[d][c] = tile rows of direction d with more than c tiles
  // (the per-warp difference arrays are free now and hold the two histograms)
  int* base = cnt_all;
  const int n1 = p.NT + 1;
  for (int x = threadIdx.x; x < 2 * n1; x += kThreads)
    base[x] = ld_acquire(&hist[x]);
  __syncthreads();
  if (warp < 2) {
    int* h = base + warp * n1;
    // suffix sums from c = NT down: lane l owns counts [NT - (l + 1) * per + 1, NT - l * per]
    const int per = (n1 + 31) >> 5;
    int run = 0;
    for (int q = 0; q < per; ++q) {
      const int c = p.NT - lane * per - q;
      if (c >= 0) run += h[c];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    int acc = incl - run;  // rows with more tiles than this lane's first count
    for (int q = 0; q < per; ++q) {
      const int c = p.NT - lane * per - q;
      if (c >= 0) {
        const int v = h[c];
        h[c] = acc;
        acc += v;
      }
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < n_items; x += kThreads) {
    const int2 it = items[x];
    if (it.x == -1) continue;
    const int d = static_cast<int>(static_cast<uint32_t>(it.x) >> 31);
    const int c = it.y >> 16, ticket = it.y & 0xFFFF;
    const int pos = base[d * n1 + c] + ticket;
    if (pos < p.B * p.NT) p.dir[d].sched[pos] = it.x & 0x7FFFFFFF;
  }
}

}  // namespace cmcore
