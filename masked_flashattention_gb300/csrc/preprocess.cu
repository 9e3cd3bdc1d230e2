// Online preprocess: evaluate compiled interval endpoints against batch metadata and emit the
// Execution Descriptor (CompileMask sections 3.3 and 3.3.1).
//
// The per-tile work (endpoints, clamping, Interval Table stores, tile classification) lives in
// descriptor_core.cuh and is shared with the mask-specific kernels generated per MaskSpec.  This
// file holds the generic kernel, whose row evaluator interprets the compiler's endpoint programs
// (one launch for both directions), the schedule kernel, and the launcher that picks one of the
// two descriptor kernels.
//
// The schedule orders tile rows longest first (LPT) for the attention kernels.
#include <cuda_runtime.h>
#include <cstdint>

#include "descriptor_core.cuh"
#include "kernels.h"
#include "program.h"

namespace cm {

constexpr int kTile = cmcore::kTile;
static_assert(cmcore::kSlots == kMaxSlots, "slot limits of the compiler and the kernel differ");

struct PrepParams {
  DevProg prog[2];           // 0: forward spec, 1: backward spec
  cmcore::DescCore core[2];  // 0: forward, 1: backward
};

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
      case OP_MODC: TOP = cmcore::imod(TOP, code[pc]); ++pc; break;
      case OP_MULC: TOP = static_cast<int>(static_cast<unsigned>(TOP) * static_cast<unsigned>(code[pc])); ++pc; break;
      case OP_NEG: TOP = static_cast<int>(0u - static_cast<unsigned>(TOP)); break;
      case OP_NOT: TOP = (TOP == 0); break;
      case OP_SEG_IDX: TOP = cmcore::seg_index(seg_s, nseg, TOP); break;
      case OP_SEG_START_AT: TOP = cmcore::seg_start_at(seg_s, nseg, TOP); break;
      case OP_SEG_END_AT: TOP = cmcore::seg_end_at(seg_s, nseg, TOP); break;
      default: {
        if (sp < 2) return 0;
        const int b = st[--sp];
        const int a = st[sp - 1];
        int r = 0;
        switch (op) {
          case OP_ADD: r = static_cast<int>(static_cast<unsigned>(a) + static_cast<unsigned>(b)); break;
          case OP_SUB: r = static_cast<int>(static_cast<unsigned>(a) - static_cast<unsigned>(b)); break;
          case OP_MIN: r = cmcore::imin(a, b); break;
          case OP_MAX: r = cmcore::imax(a, b); break;
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

// Row evaluator of the generic kernel: the first Region whose guard holds gives the row's slots.
struct InterpEval {
  const DevProg* prog;
  __device__ __forceinline__ void row(int i, int ki, const int* seg_s, int nseg, int S, int* lo,
                                      int* hi) const {
    int region = -1;
    for (int r = 0; r < prog->nreg; ++r) {
      if (eval_prog(prog->code, prog->guard[r], i, ki, seg_s, nseg, S) != 0) {
        region = r;
        break;
      }
    }
    if (region < 0) return;
#pragma unroll
    for (int n = 0; n < kMaxSlots; ++n) {
      if (n < prog->ni && n < prog->nslot[region]) {
        const int c = prog->cond[region][n];
        if (c < 0 || eval_prog(prog->code, c, i, ki, seg_s, nseg, S) != 0) {
          lo[n] = eval_prog(prog->code, prog->lo[region][n], i, ki, seg_s, nseg, S);
          hi[n] = eval_prog(prog->code, prog->hi[region][n], i, ki, seg_s, nseg, S);
        }
      }
    }
  }
};

// Both directions in one launch: block x covers tile row (x % (B*NT)) of direction x / (B*NT).
__global__ void __launch_bounds__(kTile) descriptor_kernel(const __grid_constant__ PrepParams p) {
  const int per_dir = p.core[0].B * p.core[0].NT;
  const int dir = blockIdx.x / per_dir;
  const int rem = blockIdx.x % per_dir;
  cmcore::descriptor_tile<kMaxSlots>(p.core[dir], rem / p.core[0].NT, rem % p.core[0].NT,
                                     InterpEval{&p.prog[dir]});
}

// Longest-first order of tile rows by counting sort on the number of non-empty tiles (0..NT),
// which the descriptor kernel left in the schedule array itself: the counts are staged in shared
// memory, histogrammed, scanned in descending order, and each row is placed.  Rows with equal
// counts may come in any order.  One block of 1024 threads per direction; NT <= 1024 and B * NT <= 32768.
__global__ void __launch_bounds__(1024) schedule_kernel(int32_t* sched_f, int32_t* sched_b, int B,
                                                        int NT) {
  extern __shared__ uint16_t s_cnt[];  // [B * NT]
  __shared__ int hist[1025];
  __shared__ int wsum[32];
  int32_t* sched = blockIdx.x == 0 ? sched_f : sched_b;
  const int n = B * NT;
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const unsigned full = 0xFFFFFFFFu;
  for (int c = t; c <= NT; c += blockDim.x) hist[c] = 0;
  for (int it = t; it < n; it += blockDim.x) s_cnt[it] = static_cast<uint16_t>(sched[it]);
  __syncthreads();
  for (int it = t; it < n; it += blockDim.x) atomicAdd(&hist[s_cnt[it]], 1);
  __syncthreads();
  // thread t owns count NT - t (t < NT): inclusive scan in descending count order
  const int c = NT - t;
  const int v = t < NT ? hist[c] : 0;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(full, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = wsum[lane];
    int e = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(full, e, o);
      if (lane >= o) e += y;
    }
    wsum[lane] = e - w;  // exclusive prefix of the warp totals
  }
  __syncthreads();
  const int incl = x + wsum[warp];
  __syncthreads();
  if (t < NT) hist[c] = incl - v;   // first position of count c
  if (t == NT - 1) hist[0] = incl;  // rows without tiles go last
  __syncthreads();
  for (int it = t; it < n; it += blockDim.x) {
    const int pos = atomicAdd(&hist[s_cnt[it]], 1);
    sched[pos] = ((it / NT) << 16) | (it % NT);
  }
}

int launch_descriptor(const DevProg& fwd, const DevProg& bwd, const void* gen_fwd,
                      const void* gen_bwd, const int32_t* seg, const int32_t* nseg, int nseg_max,
                      int B, int S, int32_t* itab_f, uint32_t* bm_f, int32_t* itab_b,
                      uint32_t* bm_b, int32_t* sched_f, int32_t* sched_b, int32_t* status,
                      cudaStream_t stream) {
  const int NT = S / kTile;
  const int W = (NT + 15) / 16;
  if (NT > 1024 || static_cast<long long>(B) * NT > 32768) return -1;
  const cmcore::DescCore cf{itab_f, bm_f, sched_f, seg, nseg, status, nseg_max, B, S, NT, W, fwd.ni, 0};
  const cmcore::DescCore cb{itab_b, bm_b, sched_b, seg, nseg, status, nseg_max, B, S, NT, W, bwd.ni, 1};
  const size_t smem = static_cast<size_t>(nseg_max + 1) * 4 + static_cast<size_t>(2) * (NT + 1) * 4 +
                      static_cast<size_t>(NT) + 16;
  if (smem > 200 * 1024) return -1;
  if (gen_fwd != nullptr && gen_bwd != nullptr) {
    // the mask-specific kernels: one launch per direction
    for (int dir = 0; dir < 2; ++dir) {
      const void* k = dir == 0 ? gen_fwd : gen_bwd;
      cmcore::DescCore c = dir == 0 ? cf : cb;
      if (smem > 48 * 1024 &&
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return -1;
      void* args[] = {&c};
      if (cudaLaunchKernel(k, dim3(B * NT), dim3(kTile), args, smem, stream) != cudaSuccess)
        return -1;
    }
  } else {
    PrepParams p;
    p.prog[0] = fwd;
    p.prog[1] = bwd;
    p.core[0] = cf;
    p.core[1] = cb;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(descriptor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -1;
    descriptor_kernel<<<2 * B * NT, kTile, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
  }
  const size_t sched_smem = static_cast<size_t>(B) * NT * sizeof(uint16_t);
  if (sched_smem > 48 * 1024 &&
      cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sched_smem)) != cudaSuccess)
    return -1;
  schedule_kernel<<<2, 1024, sched_smem, stream>>>(sched_f, sched_b, B, NT);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return 0;
}

}  // namespace cm
