// cz_muon_step_noalloc: the Muon step with its scratch in a static device array.
//
// Some callers cannot allocate device memory at the point where they run the
// optimizer step: a framework whose caching allocator owns all of device memory
// and forbids side allocations, a runtime that reserves memory up front and
// treats any later cudaMalloc as an error, or an embedding that must not trigger
// the implicit device synchronisation that cudaMalloc/cudaFree can cause.  For
// them this entry point runs exactly the same kernels as cz_muon_step_ex, but
// the workspace is the file-scope array below, so the call allocates nothing:
// no cudaMalloc, no cudaFree, no allocating library routine.
//
// The array holds CZ_STATIC_WORKSPACE_BYTES on every GPU that loads it, for the
// life of the process.  The CUDA runtime loads this file's module (and with it
// the array) when the module is first used on a device; under lazy module
// loading, the default, that is the first call's address look-up, so the first
// call on each device is where the driver reserves the array's memory.  Every
// call shares the array and it keeps the previous call's contents: the kernels
// overwrite everything they read except the status word, which the first call on
// a device clears on the caller's stream and cz_device_status(stream, NULL)
// reads and clears afterwards.  Calls that overlap on the GPU (different streams,
// or different host threads without ordering) race on the array.

#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "cz.h"
#include "cz_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[CZ_STATIC_WORKSPACE_BYTES];

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_ptr;   // per device: device address of g_noalloc_scratch

// Set-up, once per device, with that device current: the host name of the
// array is only a stand-in, so its device address is looked up here and passed
// on as the workspace pointer.  The status word (the first bytes of the
// workspace header) is cleared on the caller's stream, ahead of the first step's
// kernels on that stream.
int noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CZ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  auto it = g_noalloc_ptr.find(dev);
  if (it == g_noalloc_ptr.end()) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return CZ_ERR_CUDA;
    }
    if (cudaMemsetAsync(ptr, 0, 256, stream) != cudaSuccess) {
      cudaGetLastError();
      return CZ_ERR_CUDA;
    }
    it = g_noalloc_ptr.emplace(dev, ptr).first;
  }
  *out = it->second;
  return CZ_OK;
}

}  // namespace

namespace cz {

// The array's device address on the current device, or null if no
// cz_muon_step_noalloc call has set it up there (nothing is looked up or
// loaded here).
void* noalloc_scratch_if_set_up() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  auto it = g_noalloc_ptr.find(dev);
  return it == g_noalloc_ptr.end() ? nullptr : it->second;
}

}  // namespace cz

extern "C" int cz_muon_step_noalloc(const cz_plan* plan, int32_t rank, float* flat_param, const void* flat_grad,
                                    float* flat_mom, const int64_t* offsets, const int64_t* shapes, float lr,
                                    float mu, int32_t ns_steps, void* stream, const cz_step_opts* opts) {
  if (!plan || !shapes) return CZ_ERR_INVALID;
  cz_step_opts o;
  if (opts) {
    o = *opts;
    if (o.workspace || o.workspace_bytes) return CZ_ERR_INVALID;   // the scratch is the static array
  } else {
    cz_step_opts_default(&o);
  }
  // a pageable upload cannot be captured, and the first call's set-up synchronises:
  // refuse a capturing stream before anything else
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap) != cudaSuccess) {
    cudaGetLastError();
    return CZ_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return CZ_ERR_INVALID;
  size_t need = 0;
  int st = cz_workspace_size(plan, rank, shapes, &need);
  if (st != CZ_OK) return st;
  if (need > (size_t)CZ_STATIC_WORKSPACE_BYTES) return CZ_ERR_NOMEM;   // shard too large for the array
  void* scratch = nullptr;
  st = noalloc_scratch(reinterpret_cast<cudaStream_t>(stream), &scratch);
  if (st != CZ_OK) return st;
  o.workspace = scratch;
  o.workspace_bytes = (size_t)CZ_STATIC_WORKSPACE_BYTES;
  // tables stay in pageable memory: page-locking host memory can synchronise like cudaMalloc
  return cz::muon_step(plan, rank, flat_param, flat_grad, flat_mom, offsets, shapes, lr, mu, ns_steps, stream, &o,
                       false);
}
