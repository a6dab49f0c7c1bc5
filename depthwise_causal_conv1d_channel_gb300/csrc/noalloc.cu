// Backward entry point that allocates nothing.
//
// ccc_conv1d_bwd needs a caller-provided device workspace for its FP32
// weight/bias-gradient sums.  Some callers cannot provide one: code embedded in
// a host program that owns every byte of device memory and forbids allocation
// while it runs (an inference or training server with a fixed memory budget, a
// plugin interface that hands over only the operation's own tensors).  For
// them, ccc_conv1d_bwd_noalloc runs the same backward with its workspace taken
// from a fixed scratch array compiled into this library.
//
// The scratch array lives in device memory on every GPU that loads the
// library, for as long as the library stays loaded.  Its address is looked up
// once per device, on the first call made with that device current.  All calls
// on a device share the one array: calls whose work overlaps on the GPU (for
// example on two streams at once) race on it; calls on one stream are ordered
// and safe.  The backward fully writes every per-block partial row before the
// finalize kernel reads it, so stale contents from an earlier call are never
// used.
#include <atomic>
#include <mutex>

#include "ccc_conv1d.h"

namespace {

// 4 MiB: enough for the FP32 partial sums of (block rows x D) up to ~200 000.
constexpr size_t kScratchBytes = CCC_CONV1D_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) float g_bwd_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_bwd_scratch on the current device (looked up once).
ccc_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CCC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CCC_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_bwd_scratch) != cudaSuccess || addr == nullptr)
        return CCC_ERR_CUDA;
      g_scratch_addr[dev].store(addr, std::memory_order_release);
      p = addr;
    }
  }
  *out = p;
  return CCC_OK;
}

}  // namespace

extern "C" {

ccc_status ccc_conv1d_bwd_noalloc(const ccc_tensor* x, const ccc_tensor* weight,
                                  const ccc_tensor* bias, const ccc_tensor* cu_seqlens,
                                  const ccc_tensor* initial_states, const ccc_tensor* dout,
                                  const ccc_tensor* dfinal_states, const ccc_tensor* dx,
                                  const ccc_tensor* dweight, const ccc_tensor* dbias,
                                  const ccc_tensor* dinitial_states, int activation,
                                  int deterministic, int* d_status, cudaStream_t stream) {
  // 0 means x itself is rejected; ccc_conv1d_bwd then reports why.
  const size_t need = ccc_conv1d_bwd_workspace_size(x, deterministic ? 1 : 0);
  if (need > kScratchBytes) return CCC_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const ccc_status st = scratch_address(&scratch);
  if (st != CCC_OK) return st;
  return ccc_conv1d_bwd(x, weight, bias, cu_seqlens, initial_states, dout, dfinal_states, dx,
                        dweight, dbias, dinitial_states, activation, deterministic, scratch,
                        kScratchBytes, d_status, stream);
}

}  // extern "C"
