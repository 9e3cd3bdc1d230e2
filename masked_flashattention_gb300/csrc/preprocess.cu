// Online preprocess: evaluate compiled interval endpoints against batch metadata and emit the
// Execution Descriptor (CompileMask sections 3.3 and 3.3.1).
//
// One launch builds both halves.  Block x covers one 128-row tile of one sample in one direction
// (forward: query rows; backward: key columns); thread t owns row tile*128 + t:
//   1. the sample's segment boundaries are staged in shared memory and validated;
//   2. the thread picks the first Region whose guard holds and evaluates that Region's slot
//      endpoints (stack programs from the compiler), clamps them to [0, S] and stores every slot
//      as (start, end), writing (0, 0) for padding, failed conditions and empty intervals;
//      stores are 8-byte and coalesced (slot-major layout [b][slot][row]);
//   3. tile states: each row adds its touched tile ranges ("any") and the tile ranges its merged
//      intervals cover completely ("all") to two shared-memory difference arrays; a prefix sum
//      over the tiles gives, per tile, empty (no row touches it), full (all 128 rows cover it)
//      or partial.  A union of adjacent or overlapping slots counts as covering, so the states
//      equal those of the dense mask exactly.
// A second small launch orders the tile rows longest first (LPT) for the attention kernels.
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "program.h"
#include "ptx.cuh"

namespace cm {

constexpr int kTile = 128;

struct PrepParams {
  DevProg prog[2];  // 0: forward spec, 1: backward spec
  int32_t* itab[2];
  uint32_t* bm[2];
  const int32_t* seg;
  const int32_t* nseg;
  int32_t* status;
  int nseg_max;
  int B, S, NT, W;  // NT tiles per row; W = ceil(NT / 16) bitmap words per tile row
};

__device__ __forceinline__ int seg_index(const int* seg_s, int nseg, int e) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seg_s[mid] <= e) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

// Evaluate one endpoint program.  Arithmetic wraps (unsigned) instead of overflowing.
__device__ int eval_prog(const int32_t* code, int pc, int row, int row_seg, const int* seg_s,
                         int nseg, int S) {
  int st[kMaxStack];
  int sp = 0;
#define PUSH(x)                          \
  do {                                   \
    if (sp < kMaxStack) st[sp++] = (x);  \
  } while (0)
#define TOP st[sp > 0 ? sp - 1 : 0]
  for (int guard = 0; guard < kMaxCode; ++guard) {
    const int op = code[pc++];
    switch (op) {
      case OP_END: return sp > 0 ? st[sp - 1] : 0;
      case OP_CONST: PUSH(code[pc]); ++pc; break;
      case OP_I: PUSH(row); break;
      case OP_S: PUSH(S); break;
      case OP_NSEG: PUSH(nseg); break;
      case OP_SEG_IDX_I: PUSH(row_seg); break;
      case OP_MULC: TOP = static_cast<int>(static_cast<unsigned>(TOP) * static_cast<unsigned>(code[pc])); ++pc; break;
      case OP_NEG: TOP = static_cast<int>(0u - static_cast<unsigned>(TOP)); break;
      case OP_NOT: TOP = (TOP == 0); break;
      case OP_SEG_IDX: TOP = seg_index(seg_s, nseg, TOP); break;
      case OP_SEG_START_AT: TOP = seg_s[imin(imax(TOP, 0), nseg)]; break;
      case OP_SEG_END_AT: {
        const int k = TOP;
        TOP = seg_s[imin(imax(k, -1) + 1, nseg)];
        break;
      }
      default: {
        if (sp < 2) return 0;
        const int b = st[--sp];
        const int a = st[sp - 1];
        int r = 0;
        switch (op) {
          case OP_ADD: r = static_cast<int>(static_cast<unsigned>(a) + static_cast<unsigned>(b)); break;
          case OP_SUB: r = static_cast<int>(static_cast<unsigned>(a) - static_cast<unsigned>(b)); break;
          case OP_MIN: r = imin(a, b); break;
          case OP_MAX: r = imax(a, b); break;
          case OP_AND: r = (a != 0) && (b != 0); break;
          case OP_OR: r = (a != 0) || (b != 0); break;
          case OP_CMP: {
            const int c = code[pc++];
            r = c == CMP_LT ? a < b : c == CMP_LE ? a <= b : c == CMP_GT ? a > b
              : c == CMP_GE ? a >= b : c == CMP_EQ ? a == b : a != b;
            break;
          }
          default: return 0;
        }
        st[sp - 1] = r;
      }
    }
  }
#undef PUSH
#undef TOP
  return 0;
}

__global__ void __launch_bounds__(kTile) descriptor_kernel(const __grid_constant__ PrepParams p) {
  extern __shared__ int smem_i[];
  const int per_dir = p.B * p.NT;
  const int dir = blockIdx.x / per_dir;
  const int rem = blockIdx.x % per_dir;
  const int b = rem / p.NT;
  const int tile = rem % p.NT;
  const DevProg& prog = p.prog[dir];

  int* seg_s = smem_i;                         // [nseg_max + 1]
  int* cnt_any = smem_i + p.nseg_max + 1;      // [NT + 1] difference array: rows touching tile
  int* cnt_all = cnt_any + p.NT + 1;           // [NT + 1] difference array: rows covering tile
  uint8_t* code = reinterpret_cast<uint8_t*>(cnt_all + p.NT + 1);  // [NT] 2-bit state per tile
  __shared__ int s_bad;
  __shared__ int s_wtot[2][kTile / 32];

  const int t = threadIdx.x;
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
  if (s_bad && t == 0 && tile == 0) set_status(p.status, kDevBadMeta, dir);

  // --- 1. endpoints -------------------------------------------------------------------------
  const int row = tile * kTile + t;
  const int row_seg = seg_index(seg_s, nseg, row);
  int region = -1;
  for (int r = 0; r < prog.nreg; ++r) {
    if (eval_prog(prog.code, prog.guard[r], row, row_seg, seg_s, nseg, p.S) != 0) {
      region = r;
      break;
    }
  }
  int lo[kMaxSlots], hi[kMaxSlots];
#pragma unroll
  for (int n = 0; n < kMaxSlots; ++n) {
    lo[n] = 0;
    hi[n] = 0;
    if (n < prog.ni && region >= 0 && n < prog.nslot[region]) {
      const int c = prog.cond[region][n];
      if (c < 0 || eval_prog(prog.code, c, row, row_seg, seg_s, nseg, p.S) != 0) {
        int a = eval_prog(prog.code, prog.lo[region][n], row, row_seg, seg_s, nseg, p.S);
        int e = eval_prog(prog.code, prog.hi[region][n], row, row_seg, seg_s, nseg, p.S);
        a = imin(imax(a, 0), p.S);
        e = imin(imax(e, 0), p.S);
        if (e > a) {
          lo[n] = a;
          hi[n] = e;
        }
      }
    }
    if (n < prog.ni) {
      int2* dst = reinterpret_cast<int2*>(p.itab[dir]) + (static_cast<size_t>(b) * prog.ni + n) * p.S + row;
      *dst = make_int2(lo[n], hi[n]);
    }
  }

  // --- 2. merged intervals (sorted by start; overlapping or adjacent ones joined) -------------
  int ms[kMaxSlots], me[kMaxSlots];
#pragma unroll
  for (int n = 0; n < kMaxSlots; ++n) {
    ms[n] = hi[n] > lo[n] ? lo[n] : 0x7FFFFFFF;
    me[n] = hi[n];
  }
#pragma unroll
  for (int x = 0; x < kMaxSlots; ++x)
#pragma unroll
    for (int y = 0; y + 1 < kMaxSlots - x; ++y)
      if (ms[y] > ms[y + 1]) {
        int u = ms[y]; ms[y] = ms[y + 1]; ms[y + 1] = u;
        u = me[y]; me[y] = me[y + 1]; me[y + 1] = u;
      }
#pragma unroll
  for (int n = 1; n < kMaxSlots; ++n) {
    if (ms[n] != 0x7FFFFFFF && ms[n] <= me[n - 1] && ms[n - 1] != 0x7FFFFFFF) {
      ms[n] = ms[n - 1];
      me[n] = imax(me[n], me[n - 1]);
      ms[n - 1] = 0x7FFFFFFF;  // absorbed
    }
  }

  // --- 3. tile states ---------------------------------------------------------------------
  // Each row adds +1 / -1 at the ends of its touched tile ranges (any slot) and of its fully
  // covered tile ranges (merged intervals, which are disjoint, so a row counts once per tile).
  // After a prefix sum, a tile is touched by some row iff its "any" count is > 0, and full iff
  // its "all" count equals the 128 rows of the tile.
#pragma unroll
  for (int n = 0; n < kMaxSlots; ++n) {
    if (hi[n] > lo[n]) {
      atomicAdd(&cnt_any[lo[n] / kTile], 1);
      atomicAdd(&cnt_any[(hi[n] - 1) / kTile + 1], -1);
    }
    if (ms[n] != 0x7FFFFFFF) {
      const int a = (ms[n] + kTile - 1) / kTile, e = me[n] / kTile;
      if (e > a) {
        atomicAdd(&cnt_all[a], 1);
        atomicAdd(&cnt_all[e], -1);
      }
    }
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
  const int lane = t & 31, warp = t >> 5;
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
  for (int c = c0; c < c0 + per && c < p.NT; ++c) {
    run_a += cnt_any[c];
    run_f += cnt_all[c];
    code[c] = run_a > 0 ? (run_f == kTile ? 2 : 1) : 0;
  }
  __syncthreads();
  uint32_t* out = p.bm[dir] + (static_cast<size_t>(b) * p.NT + tile) * p.W;
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

// Longest-first order of tile rows by counting sort on the number of non-empty tiles (0..NT):
// histogram, descending exclusive scan, then placement.  Rows with equal counts may come in any
// order.  One block of 1024 threads per direction; NT <= 1024.
__device__ __forceinline__ int row_tile_count(const uint32_t* bm, int it, int W) {
  int c = 0;
  for (int w = 0; w < W; ++w) {
    const uint32_t x = bm[static_cast<size_t>(it) * W + w];
    c += __popc((x | (x >> 1)) & 0x55555555u);
  }
  return c;
}

__global__ void __launch_bounds__(1024) schedule_kernel(const uint32_t* bm_f, const uint32_t* bm_b,
                                                        int32_t* sched_f, int32_t* sched_b, int B,
                                                        int NT, int W) {
  __shared__ int hist[1025];
  __shared__ int wsum[32];
  const uint32_t* bm = blockIdx.x == 0 ? bm_f : bm_b;
  int32_t* sched = blockIdx.x == 0 ? sched_f : sched_b;
  const int n = B * NT;
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  for (int c = t; c <= NT; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  for (int it = t; it < n; it += blockDim.x) atomicAdd(&hist[row_tile_count(bm, it, W)], 1);
  __syncthreads();
  // thread t owns count NT - t (t < NT): inclusive scan in descending count order
  const int c = NT - t;
  const int v = t < NT ? hist[c] : 0;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
    int e = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, e, o);
      if (lane >= o) e += y;
    }
    wsum[lane] = e - w;  // exclusive prefix of the warp totals
  }
  __syncthreads();
  const int incl = x + wsum[warp];
  __syncthreads();
  if (t < NT) hist[c] = incl - v;  // first slot of count c
  if (t == NT - 1) hist[0] = incl;  // rows without tiles go last
  __syncthreads();
  for (int it = t; it < n; it += blockDim.x) {
    const int pos = atomicAdd(&hist[row_tile_count(bm, it, W)], 1);
    sched[pos] = ((it / NT) << 16) | (it % NT);
  }
}

int launch_descriptor(const DevProg& fwd, const DevProg& bwd, const int32_t* seg,
                      const int32_t* nseg, int nseg_max, int B, int S, int32_t* itab_f,
                      uint32_t* bm_f, int32_t* itab_b, uint32_t* bm_b, int32_t* sched_f,
                      int32_t* sched_b, int32_t* status, cudaStream_t stream) {
  PrepParams p;
  p.prog[0] = fwd;
  p.prog[1] = bwd;
  p.itab[0] = itab_f;
  p.itab[1] = itab_b;
  p.bm[0] = bm_f;
  p.bm[1] = bm_b;
  p.seg = seg;
  p.nseg = nseg;
  p.status = status;
  p.nseg_max = nseg_max;
  p.B = B;
  p.S = S;
  p.NT = S / kTile;
  p.W = (p.NT + 15) / 16;
  const size_t smem = static_cast<size_t>(nseg_max + 1) * 4 + static_cast<size_t>(2) * (p.NT + 1) * 4 +
                      static_cast<size_t>(p.NT) + 16;
  if (smem > 200 * 1024) return -1;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(descriptor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -1;
  }
  descriptor_kernel<<<2 * B * p.NT, kTile, smem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return -1;
  if (p.NT > 1024) return -1;
  schedule_kernel<<<2, 1024, 0, stream>>>(bm_f, bm_b, sched_f, sched_b, B, p.NT, p.W);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return 0;
}

}  // namespace cm
