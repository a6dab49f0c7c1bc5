// Single-token update (cuDNN frontend docs, "Causal Conv1d" page: the returned
// width-four final_states[B, D, 3] feed causal_conv1d_update, which mutates
// that state in place).
//
//   out[b,d]   = act(bias[d] + w0*s0 + w1*s1 + w2*s2 + w3*x[b,d])
//   state[b,d] = [s1, s2, x[b,d]]      (bitwise)
//
// One thread per V consecutive channels of one batch row: one 16-byte load of
// x, three of the state, one 16-byte store of out, three of the state.
#include "common.cuh"
#include "launch.h"

namespace ccc {

template <int V, int ACT>
__global__ void __launch_bounds__(256) update_kernel(UpdArgs a) {
  using VT = Vec<V>;
  const int groups = a.D / V;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= int64_t(a.B) * groups) return;
  const int bb = int(i / groups);
  const int d0 = int(i % groups) * V;
  float w[V][kWidth], b[V];
  load_weights<V>(a.wr, d0, w, b);
  uint16_t* s = a.state + (int64_t(bb) * a.D + d0) * kState;
  float win[kState][V], xc[V], y[V];
  load_state<V>(s, win);
  VT::unpack(VT::ld(a.x + bb * a.x_sb + d0), xc);
#pragma unroll
  for (int c = 0; c < V; ++c) {
    float p = b[c];
    p = fmaf(w[c][0], win[0][c], p);
    p = fmaf(w[c][1], win[1][c], p);
    p = fmaf(w[c][2], win[2][c], p);
    p = fmaf(w[c][3], xc[c], p);
    y[c] = act_fwd<ACT>(p);
    win[0][c] = win[1][c];
    win[1][c] = win[2][c];
    win[2][c] = xc[c];
  }
  VT::st(a.out + bb * a.o_sb + d0, VT::pack(y));
  store_state<V>(s, win);
}

cudaError_t launch_update(const UpdArgs& a, int vec, int act, cudaStream_t stream) {
  const int64_t threads = int64_t(a.B) * (a.D / vec);
  if (threads == 0) return cudaSuccess;
  const unsigned grid = unsigned((threads + 255) / 256);
  if (vec == 8) {
    if (act == kActSilu) update_kernel<8, kActSilu><<<grid, 256, 0, stream>>>(a);
    else update_kernel<8, kActNone><<<grid, 256, 0, stream>>>(a);
  } else {
    if (act == kActSilu) update_kernel<1, kActSilu><<<grid, 256, 0, stream>>>(a);
    else update_kernel<1, kActNone><<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ccc
