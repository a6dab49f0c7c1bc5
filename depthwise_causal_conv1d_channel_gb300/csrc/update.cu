// Decode update (cuDNN frontend docs, "Causal Conv1d" page: the returned
// width-four final_states[B, D, 3] feed causal_conv1d_update, which mutates
// that state in place; the commonly consumed causal-conv1d interface the page
// matches also takes L > 1 new tokens per row).  For each row, token by token:
//
//   out[b,d,l] = act(bias[d] + w0*s0 + w1*s1 + w2*s2 + w3*x[b,d,l])
//   state[b,d] <- [s1, s2, x[b,d,l]]      (bitwise)
//
// which is the forward over the L tokens with the state as initial state and
// the new state as its final state, evaluated in the same order (bitwise equal).
//
// A thread owns V consecutive channels of one or more batch rows.  With eight
// channels and a contiguous weight, each warp moves the state of its 256
// channels as one coalesced run (update_w8_kernel); otherwise each thread
// reads and writes its own channels' state directly (update_kernel).
#include "common.cuh"
#include "launch.h"

namespace ccc {

// Block (tx, ty): threadIdx.x over groups of V channels, threadIdx.y over
// groups of R batch rows.  The block stages its channels' weights once; each
// thread issues the loads of all its R rows before computing any of them.
template <int V, int ACT, int R, bool MULTI>
__global__ void __launch_bounds__(256) update_kernel(UpdArgs a) {
  const int L = MULTI ? a.L : 1;
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
        load_state2<V>(a.state, int64_t(b0 + r) * a.D + d0, a.sw, win[r]);
        xr[r] = VT::ld(a.x + int64_t(b0 + r) * a.x_sb + d0);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r >= a.B) break;
      const uint16_t* xrow = a.x + int64_t(b0 + r) * a.x_sb + d0;
      uint16_t* orow = a.out + int64_t(b0 + r) * a.o_sb + d0;
      typename VT::Raw cur = xr[r];
      for (int l = 0; l < L; ++l) {
        // the next token's load is in flight while this one is computed
        typename VT::Raw nxt = cur;
        if (l + 1 < L) nxt = VT::ld(xrow + int64_t(l + 1) * a.x_sl);
        float2 xc[H], y[H];
        VT::unpack2(cur, xc);
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
        VT::st(orow + int64_t(l) * a.o_sl, VT::pack2(y));
        cur = nxt;
      }
      store_state2<V>(a.state, int64_t(b0 + r) * a.D + d0, a.sw, win[r]);
    }
  } else {
    float w[V][kWidth], b[V];
    weights_from_smem<V>(ws, n_blk, threadIdx.x * V, w, b);
    float win[R][kState][V];
    typename VT::Raw xr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r < a.B) {
        load_state<V>(a.state, int64_t(b0 + r) * a.D + d0, a.sw, win[r]);
        xr[r] = VT::ld(a.x + int64_t(b0 + r) * a.x_sb + d0);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (b0 + r >= a.B) break;
      const uint16_t* xrow = a.x + int64_t(b0 + r) * a.x_sb + d0;
      uint16_t* orow = a.out + int64_t(b0 + r) * a.o_sb + d0;
      typename VT::Raw cur = xr[r];
      for (int l = 0; l < L; ++l) {
        typename VT::Raw nxt = cur;
        if (l + 1 < L) nxt = VT::ld(xrow + int64_t(l + 1) * a.x_sl);
        float xc[V], y[V];
        VT::unpack(cur, xc);
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
        VT::st(orow + int64_t(l) * a.o_sl, VT::pack(y));
        cur = nxt;
      }
      store_state<V>(a.state, int64_t(b0 + r) * a.D + d0, a.sw, win[r]);
    }
  }
}

// Eight-channel groups with a contiguous [D, 4] weight.  Block (32, TY): each
// warp owns 32 consecutive groups (256 channels) of R batch rows (TY = 4,
// R = 2 measured fastest at 256 x 4096: 512 blocks, all resident at once;
// 3.79 us against 4.00 for R = 1, 4.3 for R = 3, 3.85 for TY = 2).  The state
// of those channels in one row is a single contiguous run of 32 x 48 bytes;
// the warp reads and writes it as three fully used 512-byte slices and passes
// it through shared memory, where each lane takes its own 48 bytes (a
// 48-byte lane stride puts the eight lanes of each shared-memory phase on
// eight distinct 16-byte bank groups, so the exchange is conflict-free).
// Read with per-lane 48-byte strides instead, every load instruction would
// touch twice the sectors it uses.
#ifndef CCC_UPDATE_MULTI_BLOCKS
#define CCC_UPDATE_MULTI_BLOCKS 4  // resident blocks an SM asked of the L-token instance
#endif
template <int ACT, int TY, int R, bool MULTI>
__global__ void __launch_bounds__(32 * TY, MULTI ? CCC_UPDATE_MULTI_BLOCKS : 1) update_w8_kernel(UpdArgs a) {
  constexpr int kChunks = 32 * kState;  // 16-byte chunks of one warp-row of state
  __shared__ uint4 sbuf[TY][R][kChunks];
  const int lane = threadIdx.x, wy = threadIdx.y;
  const int groups = a.D / 8;
  const int g0 = blockIdx.x * 32;
  const int n_lanes = min(32, groups - g0);
  const int n_chunks = kState * n_lanes;
  const bool valid = lane < n_lanes;
  const int d0 = (g0 + lane) * 8;
  const int b0 = (blockIdx.y * blockDim.y + wy) * R;
  // L tokens a row: tokens are taken kTokChunk at a time, all loads of a chunk
  // in flight at once; the first chunk's go out with the state's
  constexpr int kTokChunk = 4;
#if CCC_PREWAIT_PREFETCH
  // the warp's state runs (16-byte aligned: D is a multiple of 8) and the x
  // rows of its first tokens, one bulk prefetch each
  if (lane < R && b0 + lane < a.B) {
    const int64_t row = b0 + lane;
    prefetch_l2_bulk(a.state + (row * a.D + int64_t(g0) * 8) * kState, uint32_t(n_chunks) * 16);
    prefetch_l2_bulk(a.x + row * a.x_sb + int64_t(g0) * 8, uint32_t(n_lanes) * 16);
  }
  if (MULTI && lane >= 1 && lane < kTokChunk && lane < a.L && b0 < a.B)
    prefetch_l2_bulk(a.x + int64_t(b0) * a.x_sb + int64_t(lane) * a.x_sl + int64_t(g0) * 8,
                     uint32_t(n_lanes) * 16);
#endif
  pdl_wait();
  pdl_release();
  if (b0 >= a.B) return;  // the whole warp: it shares b0
  float2 w[4][kWidth], bias[4];
  uint4 sr[R][kState], xr[R];
  uint4 xq[kTokChunk - 1] = {};  // tokens 1 .. kTokChunk - 1 of row b0 (MULTI, R == 1)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (b0 + r < a.B) {
      const uint4* run = reinterpret_cast<const uint4*>(a.state + (int64_t(b0 + r) * a.D + int64_t(g0) * 8) * kState);
#pragma unroll
      for (int j = 0; j < kState; ++j)
        if (lane + 32 * j < n_chunks) sr[r][j] = run[lane + 32 * j];
      if (valid) xr[r] = Vec<8>::ld(a.x + int64_t(b0 + r) * a.x_sb + d0);
    }
  }
  if constexpr (MULTI) {
    static_assert(!MULTI || R == 1, "one row a warp with L tokens");
#pragma unroll
    for (int j = 1; j < kTokChunk; ++j)
      if (valid && j < a.L) xq[j - 1] = Vec<8>::ld(a.x + int64_t(b0) * a.x_sb + int64_t(j) * a.x_sl + d0);
  }
  if (valid) weights_direct2<8>(a.wr, d0, w, bias);  // after the state loads are in flight
  if constexpr (!MULTI) {
  // Row by row: the state run of row r goes through shared memory, its output
  // and new state are computed and stored, then row r + 1, whose loads (issued
  // with row r's above) may still be landing.
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (b0 + r >= a.B) break;
#pragma unroll
    for (int j = 0; j < kState; ++j)
      if (lane + 32 * j < n_chunks) sbuf[wy][r][lane + 32 * j] = sr[r][j];
    __syncwarp();
    if (valid) {
    union { uint4 q[kState]; uint16_t h[3 * 8]; } u;
#pragma unroll
    for (int j = 0; j < kState; ++j) u.q[j] = sbuf[wy][r][kState * lane + j];
    float2 win[kState][4], xc[4], y[4];
#pragma unroll
    for (int i = 0; i < kState; ++i)
#pragma unroll
      for (int h = 0; h < 4; ++h)
        win[i][h] = make_float2(bf16_to_f32(u.h[(2 * h) * 3 + i]), bf16_to_f32(u.h[(2 * h + 1) * 3 + i]));
    Vec<8>::unpack2(xr[r], xc);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float2 p = bias[h];
      p = ffma2(w[h][0], win[0][h], p);
      p = ffma2(w[h][1], win[1][h], p);
      p = ffma2(w[h][2], win[2][h], p);
      p = ffma2(w[h][3], xc[h], p);
      y[h] = act_fwd2<ACT>(p);
    }
    Vec<8>::st(a.out + int64_t(b0 + r) * a.o_sb + d0, Vec<8>::pack2(y));
    // new state [s1, s2, x]: shift each channel's three entries down by one
    uint16_t xh[8];
    {
      union { uint4 q; uint16_t h[8]; } xv;
      xv.q = xr[r];
#pragma unroll
      for (int c = 0; c < 8; ++c) xh[c] = xv.h[c];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      u.h[c * 3 + 0] = u.h[c * 3 + 1];
      u.h[c * 3 + 1] = u.h[c * 3 + 2];
      u.h[c * 3 + 2] = xh[c];
    }
#pragma unroll
    for (int j = 0; j < kState; ++j) sbuf[wy][r][kState * lane + j] = u.q[j];
    }
    __syncwarp();
    uint4* run = reinterpret_cast<uint4*>(a.state + (int64_t(b0 + r) * a.D + int64_t(g0) * 8) * kState);
#pragma unroll
    for (int j = 0; j < kState; ++j)
      if (lane + 32 * j < n_chunks) run[lane + 32 * j] = sbuf[wy][r][lane + 32 * j];
  }
  } else {
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (b0 + r < a.B)
#pragma unroll
      for (int j = 0; j < kState; ++j)
        if (lane + 32 * j < n_chunks) sbuf[wy][r][lane + 32 * j] = sr[r][j];
  __syncwarp();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (b0 + r >= a.B || !valid) continue;
    union { uint4 q[kState]; uint16_t h[3 * 8]; } u;
#pragma unroll
    for (int j = 0; j < kState; ++j) u.q[j] = sbuf[wy][r][kState * lane + j];
    float2 win[kState][4];
#pragma unroll
    for (int i = 0; i < kState; ++i)
#pragma unroll
      for (int h = 0; h < 4; ++h)
        win[i][h] = make_float2(bf16_to_f32(u.h[(2 * h) * 3 + i]), bf16_to_f32(u.h[(2 * h + 1) * 3 + i]));
    const uint16_t* xrow = a.x + int64_t(b0 + r) * a.x_sb + d0;
    uint16_t* orow = a.out + int64_t(b0 + r) * a.o_sb + d0;
    uint4 xs[kTokChunk];
    xs[0] = xr[r];
#pragma unroll
    for (int j = 1; j < kTokChunk; ++j) xs[j] = xq[j - 1];
    for (int l0 = 0; l0 < a.L; l0 += kTokChunk) {
      // the next chunk's loads are in flight while this one is computed
      uint4 nx[kTokChunk] = {};
#pragma unroll
      for (int j = 0; j < kTokChunk; ++j) {
        const int l = l0 + kTokChunk + j;
        if (l < a.L) nx[j] = Vec<8>::ld(xrow + int64_t(l) * a.x_sl);
      }
#pragma unroll
      for (int j = 0; j < kTokChunk; ++j) {
        if (l0 + j >= a.L) break;
        float2 xc[4], y[4];
        Vec<8>::unpack2(xs[j], xc);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float2 p = bias[h];
          p = ffma2(w[h][0], win[0][h], p);
          p = ffma2(w[h][1], win[1][h], p);
          p = ffma2(w[h][2], win[2][h], p);
          p = ffma2(w[h][3], xc[h], p);
          y[h] = act_fwd2<ACT>(p);
          win[0][h] = win[1][h];
          win[1][h] = win[2][h];
          win[2][h] = xc[h];
        }
        Vec<8>::st(orow + int64_t(l0 + j) * a.o_sl, Vec<8>::pack2(y));
      }
#pragma unroll
      for (int j = 0; j < kTokChunk; ++j) xs[j] = nx[j];
    }
    // new state: the last three extended inputs, BF16 values held exactly in FP32
#pragma unroll
    for (int i = 0; i < kState; ++i)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        u.h[(2 * h) * 3 + i] = f32_to_bf16(win[i][h].x);
        u.h[(2 * h + 1) * 3 + i] = f32_to_bf16(win[i][h].y);
      }
#pragma unroll
    for (int j = 0; j < kState; ++j) sbuf[wy][r][kState * lane + j] = u.q[j];
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (b0 + r >= a.B) continue;
    uint4* run = reinterpret_cast<uint4*>(a.state + (int64_t(b0 + r) * a.D + int64_t(g0) * 8) * kState);
#pragma unroll
    for (int j = 0; j < kState; ++j)
      if (lane + 32 * j < n_chunks) run[lane + 32 * j] = sbuf[wy][r][lane + 32 * j];
  }
  }
}

#ifndef CCC_UPDATE_W8_ROWS
#define CCC_UPDATE_W8_ROWS 2  // batch rows a warp of the one-token instance
#endif
#ifndef CCC_UPDATE_W8_WARPS
#define CCC_UPDATE_W8_WARPS 4  // warps a block
#endif

template <int ACT>
static cudaError_t launch_update_w8(const UpdArgs& a, cudaStream_t stream) {
  constexpr int TY = CCC_UPDATE_W8_WARPS, R = CCC_UPDATE_W8_ROWS;
  const int64_t groups = a.D / 8;
  if (a.L == 1) {
    dim3 grid(unsigned((groups + 31) / 32), unsigned((a.B + int64_t(TY) * R - 1) / (int64_t(TY) * R)));
    return launch_kernel(update_w8_kernel<ACT, TY, R, false>, grid, dim3(32, TY), 0, stream, true, a);
  }
  constexpr int TM = 4;  // warps a block of the L-token instance (eight spill)
  dim3 grid(unsigned((groups + 31) / 32), unsigned((a.B + int64_t(TM) - 1) / int64_t(TM)));
  return launch_kernel(update_w8_kernel<ACT, TM, 1, true>, grid, dim3(32, TM), 0, stream, true, a);
}

#ifndef CCC_UPDATE_ROWS
#define CCC_UPDATE_ROWS 2
#endif
constexpr int kUpdateRows = CCC_UPDATE_ROWS;

cudaError_t launch_update(const UpdArgs& a, int vec, int act, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  if (vec == 8 && a.wr.w_vec && a.sw == kState)  // whole-warp state runs: width four
    return act == kActSilu ? launch_update_w8<kActSilu>(a, stream)
                           : launch_update_w8<kActNone>(a, stream);
  const int64_t groups = (a.D + vec - 1) / vec;
  int tx = 1;
  while (tx < groups && tx < 32) tx <<= 1;
  const int ty = 256 / tx;
  dim3 block(tx, ty);
  dim3 grid(unsigned((groups + tx - 1) / tx),
            unsigned((a.B + int64_t(ty) * kUpdateRows - 1) / (int64_t(ty) * kUpdateRows)));
  const bool multi = a.L > 1;
  auto go = [&](auto kernel) { return launch_kernel(kernel, grid, block, 0, stream, true, a); };
  constexpr int R = kUpdateRows;
  if (vec == 8) {
    if (act == kActSilu) return multi ? go(update_kernel<8, kActSilu, R, true>) : go(update_kernel<8, kActSilu, R, false>);
    return multi ? go(update_kernel<8, kActNone, R, true>) : go(update_kernel<8, kActNone, R, false>);
  }
  if (vec == 4) {
    if (act == kActSilu) return multi ? go(update_kernel<4, kActSilu, R, true>) : go(update_kernel<4, kActSilu, R, false>);
    return multi ? go(update_kernel<4, kActNone, R, true>) : go(update_kernel<4, kActNone, R, false>);
  }
  if (act == kActSilu) return multi ? go(update_kernel<1, kActSilu, R, true>) : go(update_kernel<1, kActSilu, R, false>);
  return multi ? go(update_kernel<1, kActNone, R, true>) : go(update_kernel<1, kActNone, R, false>);
}

}  // namespace ccc
