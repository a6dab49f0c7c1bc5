// Internal interface between the C-ABI layer (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace ccc {

// Launch `kernel`; with pdl, as a programmatic dependent of the previous
// kernel in the stream (it may begin before that kernel ends and must call
// pdl_wait() before reading memory that kernel could have written).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- per-context caches (context.cu) ---------------------------------------------

constexpr int kMaxDevices = 64;

// The current device and the CUDA context current on this thread (nullptr
// before the runtime has made one current).
cudaError_t current_device_context(int* dev, void** ctx);

// One value per (device, context).  get() succeeds only when the stored value
// was computed in the context current now; put() stores a value computed in
// the current context (call it after the runtime call that computed it).
class ContextCache {
 public:
  bool get(long long* value);
  void put(long long value);

 private:
  std::mutex mu_;
  void* ctx_[kMaxDevices] = {};
  long long value_[kMaxDevices] = {};
};

enum Layout { kLayoutChannelLast = 0, kLayoutTimeContiguous = 1 };

// Time-contiguous backward over pairs of channel rows (vec 16): threads per
// block, and the shortest rows that take it.
constexpr int kBdtPairThreads = 128;
constexpr int64_t kBdtPairMinTokens = 4096;

struct FwdArgs {
  const uint16_t* x;
  uint16_t* out;
  int64_t x_sb, x_sd, x_st;  // element strides of x ([B, D, T] view)
  int64_t o_sb, o_sd, o_st;
  WeightRef wr;
  const uint16_t* init;  // [S, D, sw] contiguous or nullptr
  uint16_t* fin;         // [S, D, sw] contiguous or nullptr
  int sw;                // state entries per channel: W - 1
  Seqs seqs;
  const int* ids;        // per-token sequence ids [B, T] (dense only) or nullptr
  int64_t ids_sb, ids_st;
  int B, D;
  int64_t seg_len, n_seg;  // channel-last: tokens per thread range, number of ranges
  int64_t seg_per_seq;     // dense: ranges per sequence (none straddles one), else 0
  int* status;
};

struct WgradOut {
  void* dw;          // [D, W] BF16 or FP32
  int dw_f32;
  int W;             // kernel taps 4 - W .. 3 are the weight's taps 0 .. W-1
  int64_t dw_sd, dw_sk;
  uint16_t* db;      // [D] BF16 or nullptr
  int64_t db_sd;
};

struct BwdArgs {
  const uint16_t* x;
  const uint16_t* g;   // dL/dout
  uint16_t* dx;
  int64_t x_sb, x_sd, x_st;
  int64_t g_sb, g_sd, g_st;
  int64_t dx_sb, dx_sd, dx_st;
  WeightRef wr;
  const uint16_t* init;   // [S, D, sw] or nullptr
  const uint16_t* dfin;   // [S, D, sw] or nullptr (zero gradient)
  uint16_t* dinit;        // [S, D, sw] or nullptr
  int sw;                 // state entries per channel: W - 1
  Seqs seqs;
  const int* ids;         // per-token sequence ids [B, T] (dense only) or nullptr
  int64_t ids_sb, ids_st;
  int B, D;
  int64_t seg_len, n_seg;
  int64_t seg_per_seq;    // dense: ranges per sequence (none straddles one), else 0
  float* ws;              // FP32 weight/bias-gradient partial sums, [R, D, 5]: block row r writes ws[r]
  int* status;
};


// Launch shape of one call, chosen on the host from the sizes and the SM count.
struct FwdPlan {
  int kind;      // Layout
  int ids;       // per-token sequence ids: the general kernels with id masks
  int vec;       // channels per thread (channel-last): 8 or 1
  int tx, ty;    // block shape (channel-last)
  unsigned gx, gy;
  int64_t seg_len, n_seg;
  int64_t seg_per_seq;  // dense: segments per sequence, each inside one; 0: over all tokens
  int group;     // channel-last vector forward: tokens per ring stage
};

using BwdPlan = FwdPlan;

struct UpdArgs {
  const uint16_t* x;  // [B, D, L], channel stride 1
  int64_t x_sb, x_sl;
  uint16_t* state;    // [B, D, sw] contiguous
  int sw;             // state entries per channel: W - 1
  uint16_t* out;      // [B, D, L], channel stride 1
  int64_t o_sb, o_sl;
  WeightRef wr;
  int B, D;
  int L;              // tokens per row, >= 1
};


// T_seq: the sequence length of a dense call (Q = B * T_seq), 0 for packed.
FwdPlan plan_fwd(int kind, int vec_ok, int64_t Q, int D, int64_t rows, int sm_count,
                 bool ids = false, int64_t T_seq = 0);
BwdPlan plan_bwd(int kind, int vec_ok, int64_t Q, int D, int64_t rows, int sm_count,
                 bool ids = false, int64_t T_seq = 0);
// Rows of FP32 partial sums the backward writes.
int64_t bwd_partial_rows(const BwdPlan& p, int B, bool packed);

// Tokens per ring stage of the channel-last vector forward (a multiple of 3;
// its plans cut segments in multiples of it): six, or three when a thread gets
// fewer than kFwdShortTokens tokens (the first rows are computed sooner; with
// long ranges the longer groups keep more bytes in flight).
constexpr int kFwdGroupLong = 6, kFwdGroupShort = 3;
// Threads a block of the channel-last vector forward (three blocks an SM).
// Measured with the per-sequence plan, the prefetch before the dependent
// wait and the window loaded first: 9.46 us at 4 x 2048 x 1536 against
// 9.75 us for six 128-thread blocks an SM (10.5 us for two of 384), 199.0
// against 198.8 us at 8 x 5120 x 8192, 47.7 against 47.8 us on 16 packed
// sequences.
#ifndef CCC_FWD_THREADS
#define CCC_FWD_THREADS 256
#endif
constexpr int kFwdThreads = CCC_FWD_THREADS;
// Threads a block of the channel-last vector forward with id masks (four
// blocks an SM; with seq_idx at 4 x 2048 x 1536: 13.0 us, against 13.1 us in
// two 256-thread blocks and 14.3 us in one of 512).
#ifndef CCC_FWD_IDS_THREADS
#define CCC_FWD_IDS_THREADS 128
#endif
constexpr int kFwdIdsThreads = CCC_FWD_IDS_THREADS;
constexpr int kFwdShortTokens = 48;

// Resident blocks per SM of the channel-last kernels (SiLU instance), cached.
int fwd_blocks_per_sm(int vec);
int bwd_blocks_per_sm(int vec);
// The same for the general channel-last kernels with id masks (vec 4 or 1).
int fwd_ids_blocks_per_sm(int vec);
int bwd_ids_blocks_per_sm(int vec);
// Threads per block of the general channel-last kernels.
constexpr int kGeneralThreads = 256;
// Threads per block of the channel-last backward kernel for this vector width,
// without and with id masks.
int bwd_block_threads(int vec);
int bwd_ids_block_threads(int vec);

cudaError_t launch_fwd(const FwdArgs& a, const FwdPlan& p, int act, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, const BwdPlan& p, int act, const WgradOut& o,
                       int64_t partial_rows, cudaStream_t stream);
cudaError_t launch_update(const UpdArgs& a, int vec, int act, cudaStream_t stream);

// Full-channel dilated causal conv1d (fullconv.cu).
struct FullConvArgs {
  const uint16_t* x;     // [B, T, Cin] storage: channel stride 1
  int64_t x_sb, x_st;    // element strides (multiples of 8)
  const uint16_t* w;     // packed [K, Cout, Cin] BF16, contiguous
  const void* bias;      // [Cout] BF16 or FP32, or nullptr
  int bias_f32;
  int64_t bias_s;
  uint16_t* out;         // [B, T, Cout] storage: channel stride 1
  int64_t o_sb, o_st;
  int64_t B, T;
  int Cin, Cout, K, dil;
  int* status;
};
cudaError_t launch_fullconv(const FullConvArgs& f, cudaStream_t stream);
cudaError_t launch_pack_weight(const void* w, int w_f32, int64_t s_oc, int64_t s_ic, int64_t s_k,
                               uint16_t* packed, int64_t Cout, int64_t Cin, int64_t K,
                               cudaStream_t stream);

}  // namespace ccc
