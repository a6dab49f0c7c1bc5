// Per-context caches of host-side launch facts.
//
// A kernel attribute set with cudaFuncSetAttribute, an occupancy figure, or
// the device address of a __device__ array belongs to the CUDA context the
// module was loaded in, not to the device ordinal: after cudaDeviceReset, or
// with another context made current on the same device, the module is loaded
// again.  So each cached value is stored with the context it was computed in
// and recomputed when the current context differs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "launch.h"

namespace ccc {

namespace {

PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static const PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }();
  return fn;
}

}  // namespace

cudaError_t current_device_context(int* dev, void** ctx) {
  const cudaError_t err = cudaGetDevice(dev);
  if (err != cudaSuccess) return err;
  const PFN_cuCtxGetCurrent_v4000 fn = ctx_get_current_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  CUcontext c = nullptr;
  if (fn(&c) != CUDA_SUCCESS) return cudaErrorUnknown;
  *ctx = c;
  return cudaSuccess;
}

bool ContextCache::get(long long* value) {
  int dev = -1;
  void* ctx = nullptr;
  if (current_device_context(&dev, &ctx) != cudaSuccess || ctx == nullptr) return false;
  if (dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu_);
  if (ctx_[dev] != ctx) return false;
  *value = value_[dev];
  return true;
}

void ContextCache::put(long long value) {
  int dev = -1;
  void* ctx = nullptr;
  // the runtime call that computed the value has made the context current
  if (current_device_context(&dev, &ctx) != cudaSuccess || ctx == nullptr) return;
  if (dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(mu_);
  ctx_[dev] = ctx;
  value_[dev] = value;
}

}  // namespace ccc
