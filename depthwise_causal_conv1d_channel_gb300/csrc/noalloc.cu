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
// library, for as long as the library stays loaded.  Its device address is
// looked up with cudaGetSymbolAddress on the first call made in a CUDA context
// (the array belongs to the module loaded in that context, so a new context
// on the same device -- after cudaDeviceReset, say -- gets its own lookup).
// All calls in a context share the one array: calls whose work overlaps on
// the GPU (for example on two streams at once) race on it; calls on one stream
// are ordered and safe.  The backward fully writes every per-block partial row
// before the finalize kernel reads it, so stale contents from an earlier call
// are never used.
#include "ccc_conv1d.h"
#include "launch.h"

namespace {

// 4 MiB: enough for the FP32 partial sums of (block rows x D) up to ~200 000.
constexpr size_t kScratchBytes = CCC_CONV1D_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) float g_bwd_scratch[kScratchBytes / sizeof(float)];

// Device address of g_bwd_scratch, per (device, context).
ccc::ContextCache g_scratch_addr;

// Device address of g_bwd_scratch in the current context.  In host code the
// array's name is only a host-side stand-in; the device address comes from the
// runtime, checked before use.
ccc_status scratch_address(void** out) {
  long long cached = 0;
  if (g_scratch_addr.get(&cached) && cached != 0) {
    *out = reinterpret_cast<void*>(static_cast<uintptr_t>(cached));
    return CCC_OK;
  }
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_bwd_scratch) != cudaSuccess || addr == nullptr)
    return CCC_ERR_CUDA;
  g_scratch_addr.put(static_cast<long long>(reinterpret_cast<uintptr_t>(addr)));
  *out = addr;
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
  return ccc_conv1d_bwd(x, weight, bias, cu_seqlens, nullptr, initial_states, dout, dfinal_states,
                        dx, dweight, dbias, dinitial_states, activation, deterministic, scratch,
                        kScratchBytes, d_status, stream);
}

}  // extern "C"
