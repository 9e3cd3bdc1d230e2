// C ABI of libcm.so: host-side validation and kernel launches (declarations in include/cm.h).
#include <cuda_runtime.h>
#include <cstdint>
#include <atomic>
#include <cmath>
#include <initializer_list>

#include "../../include/cm.h"
#include "kernels.h"
#include "program.h"
#include "ptx.cuh"

namespace {

constexpr int kTile = 128;
// The kernels map CTAs to (work item, head) in chunks of 128 work items with every head inside a
// chunk, in 32-bit arithmetic: 128 * H must stay below 2^31.  (No call that fits in device memory
// comes near: 2^24 heads of one 128-row tile are 0.5 TB per tensor at d = 128.)
constexpr int kMaxHeads = 1 << 24;
constexpr int kMaxS = 131072;

// which descriptor kernels cm_build_descriptor runs (cm_set_preprocess_mode)
std::atomic<int> g_preprocess_mode{CM_PREPROCESS_GENERATED};
// form of the attention kernels' partial-tile check (cm_set_interval_check)
std::atomic<int> g_interval_check{CM_CHECK_RANGE_MASK};
// limit of each bounded wait inside the attention kernels (cm_set_wait_limit_ns)
std::atomic<uint64_t> g_wait_limit_ns{cm::kDefaultWaitLimitNs};
constexpr unsigned long long kMaxWaitLimitNs = 60ull * 1000000000ull;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int S) {
  if (B < 1 || S < 1) return CM_ERR_INVALID_ARG;
  if (S % kTile != 0 || S > kMaxS) return CM_ERR_UNSUPPORTED;
  if (B > 32767 || static_cast<long long>(B) * (S / kTile) > 32768) return CM_ERR_UNSUPPORTED;
  return CM_OK;
}

int check_desc(const cm_descriptor* d, int B, int S) {
  if (!d) return CM_ERR_INVALID_ARG;
  if (d->B != B || d->S != S || d->tile != kTile) return CM_ERR_INVALID_ARG;
  if (d->form != CM_FORM_VISIBLE && d->form != CM_FORM_MASKED) return CM_ERR_INVALID_ARG;
  const int max_stored = cm::kMaxSlots + d->form;
  if (d->ni_f < 1 || d->ni_f > max_stored || d->ni_b < 1 || d->ni_b > max_stored)
    return CM_ERR_INVALID_ARG;
  if (!d->itab_f || !d->bm_f || !d->itab_b || !d->bm_b || !d->sched_f || !d->sched_b || !d->status)
    return CM_ERR_INVALID_ARG;
  if (!aligned16(d->itab_f) || !aligned16(d->itab_b)) return CM_ERR_INVALID_ARG;
  return CM_OK;
}

// Host checks shared by the attention entry points.
int check_attn(const cm_descriptor* desc, int B, int H, int S, int d, float scale) {
  int rc = check_shape(B, S);
  if (rc != CM_OK) return rc;
  rc = check_desc(desc, B, S);
  if (rc != CM_OK) return rc;
  if (H < 1 || static_cast<long long>(B) * H * (S / kTile) > 0x7FFFFFFFLL) return CM_ERR_INVALID_ARG;
  if (H > kMaxHeads) return CM_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return CM_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return CM_ERR_INVALID_ARG;
  return CM_OK;
}

// Checks of the pointers of a call (all non-null and 16-byte aligned).
int check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return CM_ERR_INVALID_ARG;
  return CM_OK;
}

size_t row_floats_bytes(int B, int H, int S) {
  const size_t rows = static_cast<size_t>(B) * H * S;
  return (rows * 4 + 255) / 256 * 256;
}

int check_workspace(const void* workspace, size_t workspace_bytes, int B, int H, int S, int d) {
  size_t need = 0;
  const int rc = cm_attn_bwd_workspace_size(B, H, S, d, &need);
  if (rc != CM_OK) return rc;
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return CM_ERR_INVALID_ARG;
  return CM_OK;
}

}  // namespace

extern "C" {

CM_API const char* cm_error_string(int code) {
  switch (code) {
    case CM_OK: return "ok";
    case CM_ERR_PARSE: return "spec does not parse or uses an unsupported form";
    case CM_ERR_INVALID_ARG: return "invalid argument";
    case CM_ERR_UNSUPPORTED: return "unsupported shape or limit";
    case CM_ERR_CUDA: return "CUDA runtime error";
    case CM_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case CM_ERR_DEVICE_CHECK: return "segment metadata failed device-side validation";
    case CM_ERR_DESC_MISMATCH:
      return "the backward Tile-State Bitmap is not the transpose of the forward one";
    default: return "unknown error";
  }
}

CM_API int cm_descriptor_sizes(const cm_spec* fwd, const cm_spec* bwd, int B, int S, int tile,
                               int form, size_t sizes[7]) {
  if (!fwd || !bwd || !sizes) return CM_ERR_INVALID_ARG;
  if (form != CM_FORM_VISIBLE && form != CM_FORM_MASKED) return CM_ERR_INVALID_ARG;
  if (tile != kTile) return CM_ERR_UNSUPPORTED;
  const int rc = check_shape(B, S);
  if (rc != CM_OK) return rc;
  const size_t NT = static_cast<size_t>(S / kTile);
  const size_t W = (NT + 15) / 16;
  // stored slots per row: the spec's interval count, or one more for the masked runs
  const size_t nif = static_cast<size_t>(cm::spec_program(fwd)->ni + form);
  const size_t nib = static_cast<size_t>(cm::spec_program(bwd)->ni + form);
  sizes[0] = static_cast<size_t>(B) * nif * S * 8;
  sizes[1] = static_cast<size_t>(B) * NT * W * 4;
  sizes[2] = static_cast<size_t>(B) * nib * S * 8;
  sizes[3] = static_cast<size_t>(B) * NT * W * 4;
  sizes[4] = static_cast<size_t>(B) * NT * 4;
  sizes[5] = static_cast<size_t>(B) * NT * 4;
  sizes[6] = static_cast<size_t>(2 + 2 * (NT + 1) + 6) * 4;  // status, barrier, histograms, queues
  return CM_OK;
}

CM_API int cm_set_interval_check(int mode) {
  if (mode != CM_CHECK_UNSIGNED && mode != CM_CHECK_TWO_COMPARE && mode != CM_CHECK_RANGE_MASK)
    return CM_ERR_INVALID_ARG;
  g_interval_check.store(mode);
  return CM_OK;
}

CM_API int cm_set_preprocess_mode(int mode) {
  if (mode != CM_PREPROCESS_GENERATED && mode != CM_PREPROCESS_GENERIC) return CM_ERR_INVALID_ARG;
  g_preprocess_mode.store(mode);
  return CM_OK;
}

CM_API int cm_build_descriptor(const cm_spec* fwd, const cm_spec* bwd, const cm_meta* meta, int B,
                               int S, cm_descriptor* desc, void* stream) {
  if (!fwd || !bwd || !meta || !meta->seg || !meta->nseg || meta->nseg_max < 1)
    return CM_ERR_INVALID_ARG;
  int rc = check_shape(B, S);
  if (rc != CM_OK) return rc;
  rc = check_desc(desc, B, S);
  if (rc != CM_OK) return rc;
  if (desc->ni_f != cm::spec_program(fwd)->ni + desc->form ||
      desc->ni_b != cm::spec_program(bwd)->ni + desc->form)
    return CM_ERR_INVALID_ARG;
  if (meta->nseg_max > 16384) return CM_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t work_bytes = static_cast<size_t>(2 + 2 * (S / kTile + 1) + 6) * 4;
  if (cudaMemsetAsync(desc->status, 0, work_bytes, st) != cudaSuccess) return CM_ERR_CUDA;
  const void* gen = g_preprocess_mode.load() == CM_PREPROCESS_GENERATED
                        ? cm::pair_generated_kernel(fwd, bwd)
                        : nullptr;
  if (cm::launch_descriptor(*cm::spec_program(fwd), *cm::spec_program(bwd), gen, meta->seg,
                            meta->nseg, meta->nseg_max, B, S, desc->itab_f, desc->bm_f,
                            desc->itab_b, desc->bm_b, desc->sched_f, desc->sched_b, desc->status,
                            desc->form, cm::kDefaultWaitLimitNs, st) != 0)
    return CM_ERR_CUDA;
  return CM_OK;
}

CM_API int cm_set_wait_limit_ns(unsigned long long ns) {
  if (ns > kMaxWaitLimitNs) return CM_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns == 0 ? cm::kDefaultWaitLimitNs : static_cast<uint64_t>(ns));
  return CM_OK;
}

CM_API int cm_attn_fwd(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                       void* o, float* lse, int B, int H, int S, int d, float scale,
                       void* stream) {
  int rc = check_attn(desc, B, H, S, d, scale);
  if (rc != CM_OK) return rc;
  rc = check_ptrs({q, k, v, o, lse});
  if (rc != CM_OK) return rc;
  cm::FwdParams p;
  p.itab = desc->itab_f;
  p.bm = desc->bm_f;
  p.sched = desc->sched_f;
  p.status = desc->status;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.S = S;
  p.NT = S / kTile;
  p.W = (p.NT + 15) / 16;
  p.NI = desc->ni_f;
  p.check = g_interval_check.load();
  p.masked = desc->form;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = g_wait_limit_ns.load();
  return cm::launch_attn_fwd(p, d, q, k, v, static_cast<cudaStream_t>(stream)) == 0
             ? CM_OK
             : CM_ERR_CUDA;
}

CM_API int cm_attn_bwd_workspace_size(int B, int H, int S, int d, size_t* bytes) {
  if (!bytes || B < 1 || H < 1 || S < 1) return CM_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CM_ERR_UNSUPPORTED;
  *bytes = 2 * row_floats_bytes(B, H, S);  // D, then LSE * log2(e)
  return CM_OK;
}

CM_API int cm_attn_bwd_prologue(const void* o, const float* lse, const void* d_o, void* workspace,
                                size_t workspace_bytes, int B, int H, int S, int d,
                                void* stream) {
  if (B < 1 || H < 1 || S < 1 || S % kTile != 0) return CM_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CM_ERR_UNSUPPORTED;
  int rc = check_ptrs({o, lse, d_o});
  if (rc != CM_OK) return rc;
  rc = check_workspace(workspace, workspace_bytes, B, H, S, d);
  if (rc != CM_OK) return rc;
  float* delta = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + row_floats_bytes(B, H, S));
  return cm::launch_bwd_prologue(d, o, d_o, lse, delta, lse2, static_cast<size_t>(B) * H * S,
                                 static_cast<cudaStream_t>(stream)) == 0
             ? CM_OK
             : CM_ERR_CUDA;
}

CM_API int cm_attn_bwd_dkdv(const cm_descriptor* desc, const void* q, const void* k,
                            const void* v, const void* d_o, void* dk, void* dv,
                            const void* workspace, size_t workspace_bytes, int B, int H, int S,
                            int d, float scale, void* stream) {
  int rc = check_attn(desc, B, H, S, d, scale);
  if (rc != CM_OK) return rc;
  rc = check_ptrs({q, k, v, d_o, dk, dv});
  if (rc != CM_OK) return rc;
  rc = check_workspace(workspace, workspace_bytes, B, H, S, d);
  if (rc != CM_OK) return rc;
  cm::BwdParams p;
  p.itab = desc->itab_b;
  p.bm = desc->bm_b;
  p.bm_f = desc->bm_f;
  p.sched = desc->sched_b;
  p.status = desc->status;
  p.lse = nullptr;
  p.delta = const_cast<float*>(static_cast<const float*>(workspace));
  p.lse2 = reinterpret_cast<float*>(const_cast<char*>(static_cast<const char*>(workspace)) +
                                    row_floats_bytes(B, H, S));
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.B = B;
  p.H = H;
  p.S = S;
  p.NT = S / kTile;
  p.W = (p.NT + 15) / 16;
  p.NI = desc->ni_b;
  p.check = g_interval_check.load();
  p.masked = desc->form;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = g_wait_limit_ns.load();
  return cm::launch_attn_dkdv(p, d, q, k, v, d_o, static_cast<cudaStream_t>(stream)) == 0
             ? CM_OK
             : CM_ERR_CUDA;
}

CM_API int cm_attn_bwd_dq(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* d_o, void* dq,
                          void* workspace, size_t workspace_bytes, int B, int H, int S, int d,
                          float scale, void* stream) {
  int rc = check_attn(desc, B, H, S, d, scale);
  if (rc != CM_OK) return rc;
  rc = check_ptrs({q, k, v, o, lse, d_o, dq});
  if (rc != CM_OK) return rc;
  rc = check_workspace(workspace, workspace_bytes, B, H, S, d);
  if (rc != CM_OK) return rc;
  cm::DqParams g;
  g.itab = desc->itab_f;
  g.bm = desc->bm_f;
  g.sched = desc->sched_f;
  g.status = desc->status;
  g.delta = static_cast<float*>(workspace);
  g.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + row_floats_bytes(B, H, S));
  g.lse = lse;
  g.o = static_cast<const __nv_bfloat16*>(o);
  g.q = static_cast<const __nv_bfloat16*>(q);
  g.d_o = static_cast<const __nv_bfloat16*>(d_o);
  g.dq = static_cast<__nv_bfloat16*>(dq);
  g.B = B;
  g.H = H;
  g.S = S;
  g.NT = S / kTile;
  g.W = (g.NT + 15) / 16;
  g.NI = desc->ni_f;
  g.check = g_interval_check.load();
  g.masked = desc->form;
  g.scale = scale;
  g.scale_log2 = scale * 1.4426950408889634f;
  g.wait_ns = g_wait_limit_ns.load();
  return cm::launch_attn_dq(g, d, k, v, static_cast<cudaStream_t>(stream)) == 0
             ? CM_OK
             : CM_ERR_CUDA;
}

CM_API int cm_attn_bwd(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, int B, int H, int S,
                       int d, float scale, void* stream) {
  // every argument is checked before the first stage is queued
  int rc = check_attn(desc, B, H, S, d, scale);
  if (rc != CM_OK) return rc;
  rc = check_ptrs({q, k, v, o, lse, d_o, dq, dk, dv});
  if (rc != CM_OK) return rc;
  rc = check_workspace(workspace, workspace_bytes, B, H, S, d);
  if (rc != CM_OK) return rc;
  // dQ first: it also writes the per-row constants that dK/dV reads
  rc = cm_attn_bwd_dq(desc, q, k, v, o, lse, d_o, dq, workspace, workspace_bytes, B, H, S, d, scale,
                      stream);
  if (rc != CM_OK) return rc;
  return cm_attn_bwd_dkdv(desc, q, k, v, d_o, dk, dv, workspace, workspace_bytes, B, H, S, d, scale,
                          stream);
}

CM_API int cm_get_status(const cm_descriptor* desc, void* stream) {
  if (!desc || !desc->status) return CM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CM_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, desc->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CM_ERR_CUDA;
  const int code = v >> 16;
  if (code == cm::kDevOk) return CM_OK;
  if (code == cm::kDevTimeout) return CM_ERR_TIMEOUT;
  if (code == cm::kDevDescMismatch) return CM_ERR_DESC_MISMATCH;
  return CM_ERR_DEVICE_CHECK;
}

}  // extern "C"
