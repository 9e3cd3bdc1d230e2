// Online preprocess: evaluate compiled interval endpoints against batch metadata and emit the
// Execution Descriptor (CompileMask sections 3.3 and 3.3.1).
//
// The whole kernel body (endpoints, clamping, Interval Table stores, tile classification, the
// longest-first schedules) lives in descriptor_core.cuh and is shared with the mask-specific
// kernels generated per pair of MaskSpecs.  This file holds the generic kernel, whose row
// evaluators interpret the compiler's endpoint programs, and the launcher: one cooperative launch
// builds both halves of the descriptor and both schedules.
#include <cuda_runtime.h>
#include <cstdint>

#include "descriptor_core.cuh"
#include "kernels.h"
#include "program.h"

namespace cm {

constexpr int kTile = cmcore::kTile;
static_assert(cmcore::kSlots == kMaxSlots, "slot limits of the compiler and the kernel differ");

struct PrepParams {
  DevProg prog[2];  // 0: forward spec, 1: backward spec
  cmcore::DescCore core;
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

// The generic kernel: both directions, both schedules, one cooperative launch.
__global__ void __launch_bounds__(cmcore::kThreads) descriptor_kernel(
    const __grid_constant__ PrepParams p) {
  cmcore::descriptor_kernel<kMaxSlots, kMaxSlots>(p.core, InterpEval{&p.prog[0]},
                                                  InterpEval{&p.prog[1]});
}

namespace {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

int launch_descriptor(const DevProg& fwd, const DevProg& bwd, const void* gen_kernel,
                      const int32_t* seg, const int32_t* nseg, int nseg_max, int B, int S,
                      int32_t* itab_f, uint32_t* bm_f, int32_t* itab_b, uint32_t* bm_b,
                      int32_t* sched_f, int32_t* sched_b, int32_t* work, int masked,
                      uint64_t wait_ns, cudaStream_t stream) {
  const int NT = S / kTile;
  const int W = (NT + 15) / 16;
  if (NT > 1024 || static_cast<long long>(B) * NT > 32768) return -1;
  const int sms = sm_count();
  if (sms <= 0) return -1;
  cmcore::DescCore c;
  c.dir[0] = cmcore::DescDir{itab_f, bm_f, sched_f, fwd.ni + masked};
  c.dir[1] = cmcore::DescDir{itab_b, bm_b, sched_b, bwd.ni + masked};
  c.seg = seg;
  c.nseg = nseg;
  c.work = work;
  c.nseg_max = nseg_max;
  c.B = B;
  c.S = S;
  c.NT = NT;
  c.W = W;
  c.groups = (NT + cmcore::kWarps - 1) / cmcore::kWarps;
  c.masked = masked;
  c.wait_ns = wait_ns;
  const int units = 2 * B * c.groups;
  const void* kernel = gen_kernel != nullptr ? gen_kernel
                                             : reinterpret_cast<const void*>(descriptor_kernel);
  // Size the shared memory for the most units a block can take when the grid is as small as it
  // can be (one block per SM), then fill every SM with as many blocks as fit at that size: every
  // block must be resident at once for the grid barrier (cooperative launch).
  const int upb_max = (units + sms - 1) / sms;
  const size_t smem = static_cast<size_t>(cmcore::smem_ints(nseg_max, NT, upb_max)) * 4;
  if (smem > 200 * 1024) return -1;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, cmcore::kThreads, smem) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  int grid = units < per_sm * sms ? units : per_sm * sms;
  c.units_per_block = (units + grid - 1) / grid;  // <= upb_max, since grid >= min(units, sms)
  grid = (units + c.units_per_block - 1) / c.units_per_block;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(cmcore::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (gen_kernel != nullptr) {
    void* args[] = {&c};
    if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) return -1;
  } else {
    PrepParams pp;
    pp.prog[0] = fwd;
    pp.prog[1] = bwd;
    pp.core = c;
    void* args[] = {&pp};
    if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) return -1;
  }
  return 0;
}

}  // namespace cm
