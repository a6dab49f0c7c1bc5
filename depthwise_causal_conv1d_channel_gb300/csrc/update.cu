// Single-token update (cuDNN frontend docs, "Causal Conv1d" page: the returned
// width-four final_states[B, D, 3] feed causal_conv1d_update, which mutates
// that state in place).
//
//   out[b,d]   = act(bias[d] + w0*s0 + w1*s1 + w2*s2 + w3*x[b,d])
//   state[b,d] = [s1, s2, x[b,d]]      (bitwise)
//
// A thread owns V consecutive channels of R batch rows: per row one 16-byte
// load of x, three of the state, one 16-byte store of out, three of the state.
#include "common.cuh"
#include "launch.h"

namespace ccc {

// Block (tx, ty): threadIdx.x over groups of V channels, threadIdx.y over
// groups of R batch rows.  The block stages its channels' weights once; each
// thread issues the loads of all its R rows before computing any of them.
template <int V, int ACT, int R>
__global__ void __launch_bounds__(256) update_kernel(UpdArgs a) {
  pdl_wait();     // the state and x may come from the previous kernel (the previous step)
  pdl_release();
  using VT = Vec<V>;
  __shared__ __align__(16) float ws[(kWidth + 1) * kMaxBlockChannels];
  const int n_blk = blockDim.x * V;
  const bool vec_w = V >= 4 && a.wr.w_vec;
  if (!vec_w) stage_weights(a.wr, blockIdx.x * n_blk, n_blk, a.D, ws);  // block-uniform
  const int d0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
  const int b0 = (blockIdx.y * blockDim.y + threadIdx.y) * R;
  if (d0 >= a.D || b0 >= a.B) return;
  if constexpr (V >= 4) {
    constexpr int H = V / 2;  // channel pairs, same arithmetic as the forward
    float2 w[H][kWidth], b[H];
    if (vec_w) weights_direct2<V>(a.wr, d0, w, b);
    else weights_from_smem2<V>(ws, n_blk, threadIdx.x * V, w, b);
    float2 win[R][kState][H];
    typename VT::Raw xr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r < a.B) {
        load_state2<V>(a.state + (int64_t(b0 + r) * a.D + d0) * kState, win[r]);
        xr[r] = VT::ld(a.x + int64_t(b0 + r) * a.x_sb + d0);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r >= a.B) break;
      float2 xc[H], y[H];
      VT::unpack2(xr[r], xc);
#pragma unroll
      for (int h = 0; h < H; ++h) {
        float2 p = b[h];
        p = ffma2(w[h][0], win[r][0][h], p);
        p = ffma2(w[h][1], win[r][1][h], p);
        p = ffma2(w[h][2], win[r][2][h], p);
        p = ffma2(w[h][3], xc[h], p);
        y[h] = act_fwd2<ACT>(p);
        win[r][0][h] = win[r][1][h];
        win[r][1][h] = win[r][2][h];
        win[r][2][h] = xc[h];
      }
      VT::st(a.out + int64_t(b0 + r) * a.o_sb + d0, VT::pack2(y));
      store_state2<V>(a.state + (int64_t(b0 + r) * a.D + d0) * kState, win[r]);
    }
  } else {
    float w[V][kWidth], b[V];
    weights_from_smem<V>(ws, n_blk, threadIdx.x * V, w, b);
    float win[R][kState][V];
    typename VT::Raw xr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r < a.B) {
        load_state<V>(a.state + (int64_t(b0 + r) * a.D + d0) * kState, win[r]);
        xr[r] = VT::ld(a.x + int64_t(b0 + r) * a.x_sb + d0);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r >= a.B) break;
      float xc[V], y[V];
      VT::unpack(xr[r], xc);
#pragma unroll
      for (int c = 0; c < V; ++c) {
        float p = b[c];
        p = fmaf(w[c][0], win[r][0][c], p);
        p = fmaf(w[c][1], win[r][1][c], p);
        p = fmaf(w[c][2], win[r][2][c], p);
        p = fmaf(w[c][3], xc[c], p);
        y[c] = act_fwd<ACT>(p);
        win[r][0][c] = win[r][1][c];
        win[r][1][c] = win[r][2][c];
        win[r][2][c] = xc[c];
      }
      VT::st(a.out + int64_t(b0 + r) * a.o_sb + d0, VT::pack(y));
      store_state<V>(a.state + (int64_t(b0 + r) * a.D + d0) * kState, win[r]);
    }
  }
}

#ifndef CCC_UPDATE_ROWS
#define CCC_UPDATE_ROWS 2
#endif
constexpr int kUpdateRows = CCC_UPDATE_ROWS;

cudaError_t launch_update(const UpdArgs& a, int vec, int act, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  const int64_t groups = (a.D + vec - 1) / vec;
  int tx = 1;
  while (tx < groups && tx < 32) tx <<= 1;
  const int ty = 256 / tx;
  dim3 block(tx, ty);
  dim3 grid(unsigned((groups + tx - 1) / tx),
            unsigned((a.B + int64_t(ty) * kUpdateRows - 1) / (int64_t(ty) * kUpdateRows)));
  if (vec == 8)
    return act == kActSilu ? launch_kernel(update_kernel<8, kActSilu, kUpdateRows>, grid, block, 0, stream, true, a)
                           : launch_kernel(update_kernel<8, kActNone, kUpdateRows>, grid, block, 0, stream, true, a);
  if (vec == 4)
    return act == kActSilu ? launch_kernel(update_kernel<4, kActSilu, kUpdateRows>, grid, block, 0, stream, true, a)
                           : launch_kernel(update_kernel<4, kActNone, kUpdateRows>, grid, block, 0, stream, true, a);
  return act == kActSilu ? launch_kernel(update_kernel<1, kActSilu, kUpdateRows>, grid, block, 0, stream, true, a)
                         : launch_kernel(update_kernel<1, kActNone, kUpdateRows>, grid, block, 0, stream, true, a);
}

}  // namespace ccc
