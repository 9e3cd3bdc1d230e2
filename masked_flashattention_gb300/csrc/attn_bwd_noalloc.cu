// Backward pass for callers that cannot allocate device memory.
//
// Some callers of this library run inside a host framework that owns all device memory and
// forbids its plugins to allocate (a fixed memory budget handed out up front), or on a
// latency-critical thread where cudaMalloc's implicit device synchronisation is not acceptable.
// They can still pass their own inputs and outputs, but not the fp32 workspace cm_attn_bwd needs
// (per-row D and LSE * log2(e)).
// cm_attn_bwd_noalloc serves them from a fixed scratch array that lives in this file's device
// module instead of a caller buffer.
//
// The scratch array is a file-scope __device__ array: every GPU that loads this module holds it
// (kNoallocScratchBytes) until the process exits.  Host code cannot use the array's name as a
// device address, so the address is looked up once per device with cudaGetSymbolAddress (with
// that device current) and cached; the first call on a device does that lookup, so it should come
// before any stream capture.  All calls share the array and it keeps the last call's contents:
// the backward's dQ kernel, which runs first, rewrites D and LSE * log2(e) of every row that the
// dK/dV kernel will read, and calls whose work overlaps on the GPU (e.g. on different streams)
// race on the array.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/cm.h"

namespace {

constexpr size_t kNoallocScratchBytes = static_cast<size_t>(CM_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's copy of g_bwd_scratch (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // reset the runtime's last-error state so later calls are not misreported
      return CM_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CM_OK;
}

}  // namespace

extern "C" {

CM_API int cm_attn_bwd_noalloc(const cm_descriptor* desc, const void* q, const void* k,
                               const void* v, const void* o, const float* lse, const void* d_o,
                               void* dq, void* dk, void* dv, int B, int H, int S, int d,
                               float scale, void* stream) {
  size_t need = 0;
  const int rc = cm_attn_bwd_workspace_size(B, H, S, d, &need);
  if (rc != CM_OK) return rc;
  if (need > kNoallocScratchBytes) return CM_ERR_UNSUPPORTED;  // problem too large for the array
  void* scratch = nullptr;
  const int rs = scratch_address(&scratch);
  if (rs != CM_OK) return rs;
  return cm_attn_bwd(desc, q, k, v, o, lse, d_o, dq, dk, dv, scratch, kNoallocScratchBytes, B, H,
                     S, d, scale, stream);
}

}  // extern "C"
