// Internal interface between the C ABI (api.cu) and the kernel translation units.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "program.h"

struct cm_spec;

namespace cm {

const DevProg* spec_program(const cm_spec* s);
// The mask-specific preprocess kernel of a (forward, backward) spec pair (a cudaKernel_t),
// compiled with NVRTC and loaded into the current context on first use; nullptr where that is
// not possible.
const void* pair_generated_kernel(const cm_spec* fwd, const cm_spec* bwd);

struct FwdParams {
  const int32_t* itab;   // forward Interval Table [B][NI][S][2]
  const uint32_t* bm;    // forward bitmaps [B][NT][W]
  const int32_t* sched;  // (b << 16 | q_tile), longest first
  int32_t* status;
  __nv_bfloat16* o;
  float* lse;
  int B, H, S, NT, W, NI;
  int check;             // form of the partial-tile check (kCheck* in mask.cuh)
  int masked;            // 1: the Interval Table holds masked intervals (their complement)
  float scale_log2;      // softmax scale * log2(e)
  uint64_t wait_ns;      // limit of each bounded wait (ns)
};

struct BwdParams {
  const int32_t* itab;   // backward Interval Table [B][NI][S][2]
  const uint32_t* bm;    // backward bitmaps [B][NT][W]
  const uint32_t* bm_f;  // forward bitmaps [B][NT][W], checked to be the transpose of bm
  const int32_t* sched;  // (b << 16 | k_tile), longest first
  int32_t* status;
  const float* lse;      // [B][H][S] natural log (forward output)
  float* delta;          // [B][H][S] -rowsum(dO * O), written by the dQ kernel (or prologue)
  float* lse2;           // [B][H][S] -LSE * log2(e) (-inf for rows that see nothing), same
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int B, H, S, NT, W, NI;
  int check;             // form of the partial-tile check (kCheck* in mask.cuh)
  int masked;            // 1: the Interval Table holds masked intervals (their complement)
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  uint64_t wait_ns;      // limit of each bounded wait (ns)
};

// dQ pass of the backward: traverses query tiles with the forward descriptor.
struct DqParams {
  const int32_t* itab;   // forward Interval Table [B][NI][S][2]
  const uint32_t* bm;    // forward bitmaps [B][NT][W]
  const int32_t* sched;  // (b << 16 | q_tile), longest first
  int32_t* status;
  float* delta;          // [B][H][S] -rowsum(dO * O), computed and written by the kernel
  float* lse2;           // [B][H][S] -LSE * log2(e), computed and written by the kernel
  const float* lse;      // [B][H][S] natural log (forward output)
  const __nv_bfloat16* o;    // forward output, read once per work item (for D)
  const __nv_bfloat16* q;    // staged once per work item by TMA, then copied into TMEM
  const __nv_bfloat16* d_o;  // staged once per work item by TMA, then copied into TMEM
  __nv_bfloat16* dq;
  int B, H, S, NT, W, NI;
  int check;             // form of the partial-tile check (kCheck* in mask.cuh)
  int masked;            // 1: the Interval Table holds masked intervals (their complement)
  float scale;
  float scale_log2;
  uint64_t wait_ns;      // limit of each bounded wait (ns)
};

// One cooperative launch that builds both halves of the descriptor and both schedules: the
// generated kernel of the (forward, backward) spec pair when gen_kernel is given, else the generic
// kernel.  `work` (zeroed by the caller) holds the status word, the grid barrier and the
// histograms of the schedule.
int launch_descriptor(const DevProg& fwd, const DevProg& bwd, const void* gen_kernel,
                      const int32_t* seg, const int32_t* nseg, int nseg_max, int B, int S,
                      int32_t* itab_f, uint32_t* bm_f, int32_t* itab_b, uint32_t* bm_b,
                      int32_t* sched_f, int32_t* sched_b, int32_t* work, int masked,
                      uint64_t wait_ns, cudaStream_t stream);
int launch_attn_fwd(const FwdParams& p, int d, const void* q, const void* k, const void* v,
                    cudaStream_t stream);
// Backward prologue: per row -D = -rowsum(dO * O) and -LSE * log2(e) (rows = B * H * S), for
// callers that run the dK/dV kernel without the dQ kernel.
int launch_bwd_prologue(int d, const void* o, const void* d_o, const float* lse, float* delta,
                        float* lse2, size_t rows, cudaStream_t stream);
// dK and dV along key tiles (backward descriptor); reads the per-row constants that the dQ
// kernel (or the prologue) wrote.
int launch_attn_dkdv(const BwdParams& p, int d, const void* q, const void* k, const void* v,
                     const void* d_o, cudaStream_t stream);
int launch_attn_dq(const DqParams& p, int d, const void* k, const void* v, cudaStream_t stream);

}  // namespace cm
