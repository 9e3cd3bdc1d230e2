// C ABI of libcm.so: host-side validation and kernel launches (declarations in include/cm.h).
#include <cuda_runtime.h>
#include <cstdint>
#include <atomic>
#include <cmath>

#include "../../include/cm.h"
#include "kernels.h"
#include "program.h"

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
std::atomic<int> g_interval_check{CM_CHECK_UNSIGNED};

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
  if (d->ni_f < 1 || d->ni_f > cm::kMaxSlots || d->ni_b < 1 || d->ni_b > cm::kMaxSlots)
    return CM_ERR_INVALID_ARG;
  if (!d->itab_f || !d->bm_f || !d->itab_b || !d->bm_b || !d->sched_f || !d->sched_b || !d->status)
    return CM_ERR_INVALID_ARG;
  if (!aligned16(d->itab_f) || !aligned16(d->itab_b)) return CM_ERR_INVALID_ARG;
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
    default: return "unknown error";
  }
}

CM_API int cm_descriptor_sizes(const cm_spec* fwd, const cm_spec* bwd, int B, int S, int tile,
                               size_t sizes[7]) {
  if (!fwd || !bwd || !sizes) return CM_ERR_INVALID_ARG;
  if (tile != kTile) return CM_ERR_UNSUPPORTED;
  const int rc = check_shape(B, S);
  if (rc != CM_OK) return rc;
  const size_t NT = static_cast<size_t>(S / kTile);
  const size_t W = (NT + 15) / 16;
  const size_t nif = static_cast<size_t>(cm::spec_program(fwd)->ni);
  const size_t nib = static_cast<size_t>(cm::spec_program(bwd)->ni);
  sizes[0] = static_cast<size_t>(B) * nif * S * 8;
  sizes[1] = static_cast<size_t>(B) * NT * W * 4;
  sizes[2] = static_cast<size_t>(B) * nib * S * 8;
  sizes[3] = static_cast<size_t>(B) * NT * W * 4;
  sizes[4] = static_cast<size_t>(B) * NT * 4;
  sizes[5] = static_cast<size_t>(B) * NT * 4;
  sizes[6] = 4;
  return CM_OK;
}

CM_API int cm_set_interval_check(int mode) {
  if (mode != CM_CHECK_UNSIGNED && mode != CM_CHECK_TWO_COMPARE && mode != CM_CHECK_MASKED)
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
  if (desc->ni_f != cm::spec_program(fwd)->ni || desc->ni_b != cm::spec_program(bwd)->ni)
    return CM_ERR_INVALID_ARG;
  if (meta->nseg_max > 16384) return CM_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(desc->status, 0, 4, st) != cudaSuccess) return CM_ERR_CUDA;
  const void* gen_f = nullptr;
  const void* gen_b = nullptr;
  if (g_preprocess_mode.load() == CM_PREPROCESS_GENERATED) {
    gen_f = cm::spec_generated_kernel(fwd);
    gen_b = gen_f != nullptr ? cm::spec_generated_kernel(bwd) : nullptr;
  }
  if (cm::launch_descriptor(*cm::spec_program(fwd), *cm::spec_program(bwd), gen_f, gen_b,
                            meta->seg, meta->nseg, meta->nseg_max, B, S, desc->itab_f, desc->bm_f,
                            desc->itab_b, desc->bm_b, desc->sched_f, desc->sched_b, desc->status,
                            st) != 0)
    return CM_ERR_CUDA;
  return CM_OK;
}

CM_API int cm_attn_fwd(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                       void* o, float* lse, int B, int H, int S, int d, float scale,
                       void* stream) {
  int rc = check_shape(B, S);
  if (rc != CM_OK) return rc;
  rc = check_desc(desc, B, S);
  if (rc != CM_OK) return rc;
  if (H < 1 || static_cast<long long>(B) * H * (S / kTile) > 0x7FFFFFFFLL) return CM_ERR_INVALID_ARG;
  if (H > kMaxHeads) return CM_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return CM_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return CM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return CM_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return CM_ERR_INVALID_ARG;
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
  p.scale_log2 = scale * 1.4426950408889634f;
  return cm::launch_attn_fwd(p, d, q, k, v, static_cast<cudaStream_t>(stream)) == 0
             ? CM_OK
             : CM_ERR_CUDA;
}

CM_API int cm_attn_bwd_workspace_size(int B, int H, int S, int d, size_t* bytes) {
  if (!bytes || B < 1 || H < 1 || S < 1) return CM_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CM_ERR_UNSUPPORTED;
  const size_t rows = static_cast<size_t>(B) * H * S;
  const size_t row_floats = (rows * 4 + 255) / 256 * 256;  // D, then LSE * log2(e)
  *bytes = 2 * row_floats;
  return CM_OK;
}

CM_API int cm_attn_bwd(const cm_descriptor* desc, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, int B, int H, int S,
                       int d, float scale, void* stream) {
  int rc = check_shape(B, S);
  if (rc != CM_OK) return rc;
  rc = check_desc(desc, B, S);
  if (rc != CM_OK) return rc;
  if (H < 1 || static_cast<long long>(B) * H * (S / kTile) > 0x7FFFFFFFLL) return CM_ERR_INVALID_ARG;
  if (H > kMaxHeads) return CM_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return CM_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv || !workspace)
    return CM_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, lse, d_o, dq, dk, dv, workspace};
  for (const void* x : ptrs)
    if (!aligned16(x)) return CM_ERR_INVALID_ARG;
  size_t need = 0;
  cm_attn_bwd_workspace_size(B, H, S, d, &need);
  if (workspace_bytes < need) return CM_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return CM_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(B) * H * S;
  const size_t row_floats = (rows * 4 + 255) / 256 * 256;
  cm::BwdParams p;
  p.itab = desc->itab_b;
  p.bm = desc->bm_b;
  p.sched = desc->sched_b;
  p.status = desc->status;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + row_floats);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.B = B;
  p.H = H;
  p.S = S;
  p.NT = S / kTile;
  p.W = (p.NT + 15) / 16;
  p.NI = desc->ni_b;
  p.check = g_interval_check.load();
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cm::launch_attn_bwd(p, d, q, k, v, o, d_o, st) != 0) return CM_ERR_CUDA;
  cm::DqParams g;
  g.itab = desc->itab_f;
  g.bm = desc->bm_f;
  g.sched = desc->sched_f;
  g.status = desc->status;
  g.delta = p.delta;
  g.lse2 = p.lse2;
  g.dq = static_cast<__nv_bfloat16*>(dq);
  g.B = B;
  g.H = H;
  g.S = S;
  g.NT = p.NT;
  g.W = p.W;
  g.NI = desc->ni_f;
  g.check = p.check;
  g.scale = scale;
  g.scale_log2 = p.scale_log2;
  return cm::launch_attn_dq(g, d, q, k, v, d_o, st) == 0 ? CM_OK : CM_ERR_CUDA;
}

CM_API int cm_get_status(const cm_descriptor* desc, void* stream) {
  if (!desc || !desc->status) return CM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CM_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, desc->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CM_ERR_CUDA;
  const int code = v >> 16;
  if (code == 0) return CM_OK;
  if (code == 1) return CM_ERR_TIMEOUT;
  return CM_ERR_DEVICE_CHECK;
}

}  // extern "C"
