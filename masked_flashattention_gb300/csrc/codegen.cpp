// Run-time compilation of mask-specific preprocess kernels.
//
// CompileMask compiles each MaskSpec into a mask-specific preprocess kernel (section 3.1).  The
// compiler (compiler.cpp) emits the spec's row evaluator as CUDA C++.  Here NVRTC compiles that
// source for sm_103a, together with the shared kernel body (descriptor_core.cuh, embedded in the
// library at build time), and the cubin is loaded as a CUDA library.  NVRTC is opened with
// dlopen, so a process without it still works: the generic kernel, which interprets the same
// endpoint programs on the GPU, builds the identical descriptor instead.
#include <dlfcn.h>
#include <cuda_runtime.h>
#include <nvrtc.h>

#include <string>
#include <vector>

#include "cm.h"

namespace cm {
namespace {

const char* kCoreSrc =
#include "descriptor_core_src.inc"
    ;

struct Nvrtc {
  decltype(&nvrtcCreateProgram) create = nullptr;
  decltype(&nvrtcCompileProgram) compile = nullptr;
  decltype(&nvrtcGetCUBINSize) cubin_size = nullptr;
  decltype(&nvrtcGetCUBIN) cubin = nullptr;
  decltype(&nvrtcGetProgramLogSize) log_size = nullptr;
  decltype(&nvrtcGetProgramLog) log = nullptr;
  decltype(&nvrtcDestroyProgram) destroy = nullptr;
  bool ok = false;
};

Nvrtc open_nvrtc() {
  Nvrtc n;
  void* h = nullptr;
  for (const char* name : {"libnvrtc.so.13", "libnvrtc.so", "/usr/local/cuda/lib64/libnvrtc.so.13"}) {
    h = dlopen(name, RTLD_NOW | RTLD_LOCAL);
    if (h) break;
  }
  if (!h) return n;
  n.create = reinterpret_cast<decltype(&nvrtcCreateProgram)>(dlsym(h, "nvrtcCreateProgram"));
  n.compile = reinterpret_cast<decltype(&nvrtcCompileProgram)>(dlsym(h, "nvrtcCompileProgram"));
  n.cubin_size = reinterpret_cast<decltype(&nvrtcGetCUBINSize)>(dlsym(h, "nvrtcGetCUBINSize"));
  n.cubin = reinterpret_cast<decltype(&nvrtcGetCUBIN)>(dlsym(h, "nvrtcGetCUBIN"));
  n.log_size = reinterpret_cast<decltype(&nvrtcGetProgramLogSize)>(dlsym(h, "nvrtcGetProgramLogSize"));
  n.log = reinterpret_cast<decltype(&nvrtcGetProgramLog)>(dlsym(h, "nvrtcGetProgramLog"));
  n.destroy = reinterpret_cast<decltype(&nvrtcDestroyProgram)>(dlsym(h, "nvrtcDestroyProgram"));
  n.ok = n.create && n.compile && n.cubin_size && n.cubin && n.log_size && n.log && n.destroy;
  return n;
}

const Nvrtc& nvrtc() {
  static const Nvrtc n = open_nvrtc();
  return n;
}

}  // namespace

// Compile `source` (which includes "descriptor_core.cuh") to an sm_103a cubin.  Returns CM_OK,
// CM_ERR_UNSUPPORTED (no NVRTC) or CM_ERR_CUDA (compilation failed; the log says why).
int compile_generated_kernel(const std::string& source, std::vector<char>* cubin,
                             std::string* log) {
  const Nvrtc& nv = nvrtc();
  if (!nv.ok) {
    if (log) *log = "NVRTC (libnvrtc.so.13) could not be opened";
    return CM_ERR_UNSUPPORTED;
  }
  nvrtcProgram prog = nullptr;
  const char* headers[] = {kCoreSrc};
  const char* names[] = {"descriptor_core.cuh"};
  if (nv.create(&prog, source.c_str(), "cm_generated_descriptor.cu", 1, headers, names) !=
      NVRTC_SUCCESS) {
    if (log) *log = "nvrtcCreateProgram failed";
    return CM_ERR_CUDA;
  }
  const char* opts[] = {"--gpu-architecture=sm_103a", "-std=c++17"};
  const nvrtcResult rc = nv.compile(prog, 2, opts);
  size_t log_n = 0;
  if (log && nv.log_size(prog, &log_n) == NVRTC_SUCCESS && log_n > 1) {
    log->assign(log_n, '\0');
    nv.log(prog, &(*log)[0]);
    log->resize(log_n - 1);
  }
  bool ok = rc == NVRTC_SUCCESS;
  size_t n = 0;
  if (ok && nv.cubin_size(prog, &n) == NVRTC_SUCCESS && n > 0) {
    cubin->resize(n);
    ok = nv.cubin(prog, cubin->data()) == NVRTC_SUCCESS;
  } else {
    ok = false;
  }
  nv.destroy(&prog);
  if (!ok && log && log->empty()) *log = "NVRTC compilation failed";
  return ok ? CM_OK : CM_ERR_CUDA;
}

// Compile the generated kernel and load it into the current device context.  On success
// *kernel is a cudaKernel_t, usable as the function of cudaLaunchKernel; the CUDA library stays
// loaded for the life of the process.
int load_generated_kernel(const std::string& source, const void** kernel, std::string* log) {
  *kernel = nullptr;
  std::vector<char> cubin;
  const int rc = compile_generated_kernel(source, &cubin, log);
  if (rc != CM_OK) return rc;
  cudaLibrary_t lib = nullptr;
  cudaError_t e = cudaLibraryLoadData(&lib, cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (log) *log = std::string("cudaLibraryLoadData: ") + cudaGetErrorString(e);
    return CM_ERR_CUDA;
  }
  cudaKernel_t k = nullptr;
  e = cudaLibraryGetKernel(&k, lib, "cm_generated_descriptor");
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (log) *log = std::string("cudaLibraryGetKernel: ") + cudaGetErrorString(e);
    return CM_ERR_CUDA;
  }
  *kernel = reinterpret_cast<const void*>(k);
  return CM_OK;
}

}  // namespace cm
