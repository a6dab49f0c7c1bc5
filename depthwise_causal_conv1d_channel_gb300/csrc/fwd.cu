// Forward kernels of the depthwise causal conv1d (cuDNN frontend docs, "Causal
// Conv1d" page: BF16 activations, width four, SiLU, W-1 initial and final
// state, dense or cu_seqlens-packed).
//
// Each thread owns V consecutive channels and walks a contiguous range of
// tokens, keeping the last three inputs of every channel in registers, so each
// input is read from HBM once (plus a three-token halo per range) and each
// output written once.  Nothing is staged: the op is a streaming stencil with
// about one FLOP per byte, bound by HBM bandwidth, not a contraction.  The
// weights are held halved, so the sums below are h = pre / 2 (see the
// activation section of common.cuh).
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace ccc {

// One thread: channels [d0, d0 + V), tokens [q, q_end) of one token stream.
// `n_base` is the state index of the stream's sequence 0.  U token loads are
// in flight per step; rows P tokens further on are prefetched into L2 (P = 0:
// none), so the bytes in flight do not depend on registers.  With IDS, every
// token carries a sequence id (cuDNN page, seq_idx[B, T]): a tap reads a window
// token of another id as zero.
template <int V, int ACT, int U, int P, bool IDS = false>
__device__ __forceinline__ void fwd_walk(const FwdArgs& a, const Seqs& seqs, const Stream& xs,
                                         const Stream& os, int n_base, int d0,
                                         const float (&w)[V][kWidth], const float (&b)[V],
                                         int64_t q, int64_t q_end) {
  using VT = Vec<V>;
  int n = find_seq(seqs, q);
  while (q < q_end) {
    int64_t lo, hi;
    seq_bounds(seqs, n, lo, hi);
    const int64_t e = q_end < hi ? q_end : hi;
    const int64_t state_row = (int64_t(n_base) + n) * a.D + d0;

    // win[j] = xe[q - 3 + j]: from x, or from the initial state before the
    // sequence start, or zero.
    float win[kState][V];
    // ids of the window tokens (IDS; before the row start the window is zero,
    // so any id serves), and the element offset of token t's id: id_off + t * ids_st
    int iw[kState] = {0, 0, 0};
    const int64_t id_off = IDS ? (int64_t(n_base) + n) * a.ids_sb - lo * a.ids_st : 0;
    {
      float init[kState][V];
      if (q - kState < lo && a.init) {
        load_state<V>(a.init, state_row, a.sw, init);
      } else {
#pragma unroll
        for (int i = 0; i < kState; ++i)
#pragma unroll
          for (int c = 0; c < V; ++c) init[i][c] = 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kState; ++j) {
        const int64_t tok = q - kState + j;
        if (tok >= lo) {
          VT::unpack(VT::ld(a.x + xs.at(n, tok)), win[j]);
          if constexpr (IDS) iw[j] = __ldg(a.ids + id_off + tok * a.ids_st);
        } else {
          const int64_t i = tok - lo + kState;  // 0..2
#pragma unroll
          for (int c = 0; c < V; ++c)
            win[j][c] = i == 0 ? init[0][c] : (i == 1 ? init[1][c] : init[2][c]);
        }
      }
    }

    auto step = [&](typename VT::Raw raw, int64_t t) {
      float cur[V], y[V];
      VT::unpack(raw, cur);
      bool m0 = true, m1 = true, m2 = true;  // window token k feeds token t
      if constexpr (IDS) {
        const int cid = __ldg(a.ids + id_off + t * a.ids_st);
        m0 = iw[0] == cid;
        m1 = iw[1] == cid;
        m2 = iw[2] == cid;
        iw[0] = iw[1];
        iw[1] = iw[2];
        iw[2] = cid;
      }
#pragma unroll
      for (int c = 0; c < V; ++c) {
        float p = b[c];
        p = fmaf(w[c][0], m0 ? win[0][c] : 0.0f, p);
        p = fmaf(w[c][1], m1 ? win[1][c] : 0.0f, p);
        p = fmaf(w[c][2], m2 ? win[2][c] : 0.0f, p);
        p = fmaf(w[c][3], cur[c], p);
        y[c] = act_fwd<ACT>(p);
        win[0][c] = win[1][c];
        win[1][c] = win[2][c];
        win[2][c] = cur[c];
      }
      VT::st(a.out + os.at(n, t), VT::pack(y));
    };

    if constexpr (P > 0) {
      for (int64_t t = q + U; t < q + U + P && t < e; ++t) prefetch_l2(a.x + xs.at(n, t));
    }
    // steady state: U loads in flight, then U outputs
    for (; q + U <= e; q += U) {
      if constexpr (P > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t t = q + U + P + u;
          if (t < e) prefetch_l2(a.x + xs.at(n, t));
        }
      }
      typename VT::Raw raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) raw[u] = VT::ld(a.x + xs.at(n, q + u));
#pragma unroll
      for (int u = 0; u < U; ++u) step(raw[u], q + u);
    }
    for (; q < e; ++q) step(VT::ld(a.x + xs.at(n, q)), q);

    // the thread that finishes a sequence writes its final state: xe[len-3 .. len-1]
    // (from a copy: the window's own address never leaves this function, so it
    // stays in registers, though narrow states go through an out-of-line store)
    if (e == hi && a.fin) {
      float fin[kState][V];
#pragma unroll
      for (int i = 0; i < kState; ++i)
#pragma unroll
        for (int c = 0; c < V; ++c) fin[i][c] = win[i][c];
      store_state<V>(a.fin, state_row, a.sw, fin);
    }
    ++n;
  }
}

// Channel-last x ([B, T, D] storage seen as [B, D, T]; stride of D is 1).
// Block (TX, TY): threadIdx.x runs over groups of V channels, threadIdx.y over
// token ranges of seg_len tokens.  A warp reads 32 * V * 2 contiguous bytes
// per token.
template <int V, int ACT, bool IDS = false>
__global__ void __launch_bounds__(kGeneralThreads) fwd_cl_kernel(FwdArgs a) {
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_release();
  __shared__ __align__(16) float ws[(kWidth + 1) * kMaxBlockChannels];
  if (block_rejects_cu_seqlens(a.seqs, a.status)) return;
  const int n_blk = blockDim.x * V;
  stage_weights(a.wr, blockIdx.x * n_blk, n_blk, a.D, ws);
  const int d0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
  const int64_t seg = int64_t(blockIdx.y) * blockDim.y + threadIdx.y;
  if (d0 >= a.D || seg >= a.n_seg) return;
  float w[V][kWidth], b[V];
  weights_from_smem<V>(ws, n_blk, threadIdx.x * V, w, b);
  int64_t q0, q1;
  seg_range(a.seqs, seg, a.seg_len, a.seg_per_seq, q0, q1);
  const bool dense = a.seqs.cu == nullptr;
  const Stream xs{d0, dense ? a.x_sb - a.seqs.T * a.x_st : 0, a.x_st};
  const Stream os{d0, dense ? a.o_sb - a.seqs.T * a.o_st : 0, a.o_st};
  fwd_walk<V, ACT, 4, (V == 8 ? 16 : 0), IDS>(a, a.seqs, xs, os, 0, d0, w, b, q0, q1);
}

// Channel-last x with vectors of V = 4 channels, computed as two channel
// pairs of scalar instructions (the fast path; eight channels a thread, two
// blocks per SM, measured slower, paired instructions 1-2% slower).  Same
// walk as fwd_walk, specialised: the three-token window lives in three register
// slots that rotate (the newest token overwrites the oldest slot), so full
// groups of kFwdGroup tokens (a multiple of three) need no register copies.
// The x rows stream through the thread's own ring of kFwdRing stages of one
// group each in shared memory, filled with cp.async kFwdRing - 1 groups ahead
// of the group being computed: no step waits on a load it has just issued, and
// no registers are held by loads in flight.  Segments are planned in multiples
// of kFwdGroup tokens, so only a sequence's last group can be partial; its
// tokens take the physically shifting step from the same ring.
constexpr int kFwdGroup = kFwdGroupLong;  // tokens per ring stage (multiple of 3)
#ifndef CCC_FWD_RING
#define CCC_FWD_RING 4
#endif
constexpr int kFwdRing = CCC_FWD_RING;
static_assert(kFwdRing >= 2, "the ring needs a stage being filled and one being read");
template <int V>
constexpr size_t fwd_ring_bytes(int threads, int group = kFwdGroup) {
  return size_t(threads) * kFwdRing * group * (2 * V);
}
extern __shared__ __align__(16) char fwd_dyn_smem[];

// With IDS, every token carries a sequence id (cuDNN page, seq_idx[B, T]; dense
// calls without states): a tap reads a window token of another id as zero.
// The ids of a ring group are loaded (one 4-byte load per token, the same
// address for all lanes of a warp) before the wait for the group's rows.  A
// group whose tokens and the three before them share one id (all but the
// groups at an id change, for ids that form runs) takes the unmasked steps;
// any other takes the masked step with physical shifts.  A group is a whole
// number of window periods, so both leave the window at phase 0.
#ifndef CCC_FWD_IDS_BLOCKS
#define CCC_FWD_IDS_BLOCKS 4  // resident blocks an SM asked of the id instance
#endif
template <bool IDS>
__host__ __device__ constexpr int fwd_threads() { return IDS ? kFwdIdsThreads : kFwdThreads; }
// W3: a contiguous [D, 3] weight read with vectors (its own instance, so the
// width-four kernel's register allocation is untouched).
template <int V, int ACT, bool IDS = false, bool W3 = false, int GT = kFwdGroup>
__global__ void __launch_bounds__(fwd_threads<IDS>(), IDS ? CCC_FWD_IDS_BLOCKS : 3 * 256 / kFwdThreads)
    fwd_clv_kernel(FwdArgs a) {
  constexpr int NT = fwd_threads<IDS>();
  if (blockDim.x * blockDim.y * blockDim.z != NT) return;  // the ring layout assumes it
  using VT = Vec<V>;
  using Raw = typename VT::Raw;
  constexpr int H = V / 2;  // channel pairs
  constexpr int RB = int(sizeof(Raw));
  constexpr int G = GT;
#if CCC_PREWAIT_PREFETCH
  // dense calls: the rows of the first ring groups and the three before them
  // (measured: dense_state shape 11.9 -> 10.6 us, with seq_idx 15.2 -> 13.4 us;
  // packed calls, whose first loads are a smaller share, 48.5 -> 48.7 us)
  if (a.seqs.cu == nullptr) {
    const int d0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
    const int64_t seg = int64_t(blockIdx.y) * blockDim.y + threadIdx.y;
    if (d0 < a.D && seg < a.n_seg) {
      int64_t q, q_end;
      seg_range(a.seqs, seg, a.seg_len, a.seg_per_seq, q, q_end);
      const int n = find_seq(a.seqs, q);
      const int64_t t = q - int64_t(n) * a.seqs.T;  // token within its sequence
      const int rows = int(min(min(q_end - q, int64_t((kFwdRing - 1) * G)), a.seqs.T - t));
      const uint16_t* xp = a.x + int64_t(n) * a.x_sb + t * a.x_st + d0;
      for (int u = t < kState ? -int(t) : -kState; u < rows; ++u) prefetch_l2(xp + u * a.x_st);
    }
  }
#endif
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_release();
  static_assert(G % 3 == 0, "a group is a whole number of window periods");
  __shared__ __align__(16) float ws[(kWidth + 1) * kMaxBlockChannels];
  if (block_rejects_cu_seqlens(a.seqs, a.status)) return;
  const int n_blk = blockDim.x * V;
  const int d0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
  const int64_t seg = int64_t(blockIdx.y) * blockDim.y + threadIdx.y;
  if (!a.wr.w_vec && !W3) stage_weights(a.wr, blockIdx.x * n_blk, n_blk, a.D, ws);  // block-uniform
  if (d0 >= a.D || seg >= a.n_seg) return;
  float2 w[H][kWidth], b[H];
  bool have_w = false;  // the weights are loaded once the first ring groups are in flight
  // this thread's ring: slot (stage, row u) at byte ((stage * G + u) * NT + tid) * RB
  // (a compile-time block size: the offsets are immediates)
  const int tid = threadIdx.y * blockDim.x + threadIdx.x;
  const char* ring = fwd_dyn_smem + size_t(tid) * RB;
  const uint32_t ring_s = smem_u32(ring);
  constexpr uint32_t slot = uint32_t(NT) * RB;

  int64_t q, q_end;
  seg_range(a.seqs, seg, a.seg_len, a.seg_per_seq, q, q_end);
  const bool dense = a.seqs.cu == nullptr;
  int n = find_seq(a.seqs, q);
  using P0 = std::integral_constant<int, 0>;
  using P1 = std::integral_constant<int, 1>;
  using P2 = std::integral_constant<int, 2>;
  while (q < q_end) {
    int64_t lo, hi;
    seq_bounds(a.seqs, n, lo, hi);
    const int64_t e = q_end < hi ? q_end : hi;
    const int64_t state_row = int64_t(n) * a.D + d0;
    // pointers at token q
    const uint16_t* xp = a.x + (dense ? n * a.x_sb + (q - lo) * a.x_st : q * a.x_st) + d0;
    uint16_t* op = a.out + (dense ? n * a.o_sb + (q - lo) * a.o_st : q * a.o_st) + d0;
    const int64_t xst = a.x_st, ost = a.o_st;
    const int n_tok = int(e - q);  // a segment's tokens: below 2^31
    const int n_grp = (n_tok + G - 1) / G;  // the last one may be partial

    // group k: rows q + kG .. q + kG + G - 1 (those below e) into stage k % kFwdRing
    auto issue = [&](int k) {
      const uint32_t s0 = ring_s + uint32_t((k % kFwdRing) * G) * slot;
      const uint16_t* xm = xp + int64_t(k) * G * xst;
      if (k * G + G <= n_tok) {
#pragma unroll
        for (int u = 0; u < G; ++u) cp_async<RB>(s0 + uint32_t(u) * slot, xm + u * xst);
      } else {
#pragma unroll
        for (int u = 0; u < G; ++u)
          if (k * G + u < n_tok) cp_async<RB>(s0 + uint32_t(u) * slot, xm + u * xst);
      }
    };

    // W[j] = xe[q - 3 + j]; IW[j] = its id (IDS; any value before the row
    // start, where the window is zero)
    float2 W[kState][H];
    int IW[kState] = {0, 0, 0};
    const int64_t id_off = IDS ? int64_t(n) * a.ids_sb - lo * a.ids_st : 0;
    {
      // With short ranges (3-token groups) or id masks, the window's own loads
      // (the halo rows, or the initial state) and the weights go out before
      // the ring's first groups: the first step needs them all, and requests
      // are served about in the order issued.  Measured at 4 x 2048 x 1536:
      // 10.2 -> 9.75 us, width three 10.14 -> 9.68 us, with seq_idx 13.0 ->
      // 12.64 us.  Long ranges keep the ring first (8 x 5120 x 8192 took
      // 198.5 us this way against 201.3 us the other way, 16 packed sequences
      // 47.8 against 48.1 us; holding the halo rows raw until the ring is out
      // took them from 199.5 and 48.6 us).
      float2 init[kState][H];
      if (q - kState < lo && a.init) {
        load_state2<V>(a.init, state_row, a.sw, init);
      } else {
#pragma unroll
        for (int i = 0; i < kState; ++i)
#pragma unroll
          for (int h = 0; h < H; ++h) init[i][h] = splat2(0.0f);
      }
      Raw hx[kState] = {};  // halo rows
      auto load_halo = [&]() {
#pragma unroll
        for (int j = 0; j < kState; ++j)
          if (q - kState + j >= lo) hx[j] = VT::ld(xp - (kState - j) * xst);
      };
      auto load_weights = [&]() {
        if (!have_w) {
          if constexpr (W3) weights_direct3<V>(a.wr, d0, w, b);
          else if (a.wr.w_vec) weights_direct2<V>(a.wr, d0, w, b);
          else weights_from_smem2<V>(ws, n_blk, threadIdx.x * V, w, b);
          have_w = true;
        }
      };
      auto issue_first = [&]() {
#pragma unroll
        for (int k = 0; k < kFwdRing - 1; ++k) {
          if (k < n_grp) issue(k);
          cp_async_commit();
        }
      };
      if constexpr (G == kFwdGroupShort || IDS) {
        load_halo();
        load_weights();
        issue_first();
      } else {
        issue_first();
        load_weights();
        load_halo();
      }
#pragma unroll
      for (int j = 0; j < kState; ++j) {
        const int64_t tok = q - kState + j;
        if (tok >= lo) {
          VT::unpack2(hx[j], W[j]);
          if constexpr (IDS) IW[j] = __ldg(a.ids + id_off + tok * a.ids_st);
        } else {
          const int64_t i = tok - lo + kState;
#pragma unroll
          for (int h = 0; h < H; ++h)
            W[j][h] = i == 0 ? init[0][h] : (i == 1 ? init[1][h] : init[2][h]);
        }
      }
    }
    const float2 zero2 = splat2(0.0f);

    // one token at window phase J: taps W[J], W[J+1], W[J+2] (mod 3), then the
    // new token replaces W[J]
    auto step = [&](auto phase, Raw raw, uint16_t* dst) {
      constexpr int J = decltype(phase)::value;
      float2 cur[H], y[H];
      VT::unpack2(raw, cur);
#pragma unroll
      for (int h = 0; h < H; ++h) {
        float2 p = b[h];
        p = ffma2_split(w[h][0], W[J][h], p);
        p = ffma2_split(w[h][1], W[(J + 1) % 3][h], p);
        p = ffma2_split(w[h][2], W[(J + 2) % 3][h], p);
        p = ffma2_split(w[h][3], cur[h], p);
        y[h] = act_fwd2<ACT, true>(p);
        W[J][h] = cur[h];
      }
      VT::st(dst, VT::pack2(y));
    };
    // one token with a physical shift (keeps the window at phase 0); cid is
    // its id (IDS)
    auto shift_step = [&](Raw raw, int cid, uint16_t* dst) {
      bool m0 = true, m1 = true, m2 = true;
      if constexpr (IDS) {
        m0 = IW[0] == cid;
        m1 = IW[1] == cid;
        m2 = IW[2] == cid;
        IW[0] = IW[1];
        IW[1] = IW[2];
        IW[2] = cid;
      }
      float2 cur[H], y[H];
      VT::unpack2(raw, cur);
#pragma unroll
      for (int h = 0; h < H; ++h) {
        float2 p = b[h];
        p = ffma2_split(w[h][0], m0 ? W[0][h] : zero2, p);
        p = ffma2_split(w[h][1], m1 ? W[1][h] : zero2, p);
        p = ffma2_split(w[h][2], m2 ? W[2][h] : zero2, p);
        p = ffma2_split(w[h][3], cur[h], p);
        y[h] = act_fwd2<ACT, true>(p);
        W[0][h] = W[1][h];
        W[1][h] = W[2][h];
        W[2][h] = cur[h];
      }
      VT::st(dst, VT::pack2(y));
    };

    for (int k = 0; k < n_grp; ++k) {
      if (k + kFwdRing - 1 < n_grp) issue(k + kFwdRing - 1);
      cp_async_commit();
      // one id over the group and the window before it (IDS)?
      bool uniform = true;
      if constexpr (IDS) {
        uniform = IW[0] == IW[1] && IW[1] == IW[2];
#pragma unroll
        for (int u = 0; u < G; ++u) {
          const int64_t t = q + int64_t(k) * G + u;
          if (t < e) uniform = uniform && __ldg(a.ids + id_off + t * a.ids_st) == IW[2];
        }
      }
      cp_async_wait<kFwdRing - 1>();  // group k has landed
      const char* s0 = ring + size_t((k % kFwdRing) * G) * slot;
      Raw r[G];
#pragma unroll
      for (int u = 0; u < G; ++u) r[u] = *reinterpret_cast<const Raw*>(s0 + size_t(u) * slot);
      uint16_t* om = op + int64_t(k) * G * ost;
      if (k * G + G <= n_tok && uniform) {
#pragma unroll
        for (int u = 0; u < G; u += 3) {
          step(P0{}, r[u], om + u * ost);
          step(P1{}, r[u + 1], om + (u + 1) * ost);
          step(P2{}, r[u + 2], om + (u + 2) * ost);
        }
      } else {
#pragma unroll
        for (int u = 0; u < G; ++u)
          if (k * G + u < n_tok)
            shift_step(r[u], IDS ? __ldg(a.ids + id_off + (q + int64_t(k) * G + u) * a.ids_st) : 0,
                       om + u * ost);
      }
    }
    if (e == hi && a.fin) store_state2<V>(a.fin, state_row, a.sw, W);
    q = e;
    ++n;
  }
}

// Time-contiguous x, dense, T a multiple of 8 and 16-byte aligned rows (the
// usual contiguous [B, D, T] tensor).  One warp per (batch, channel) row; each
// lane takes 8 consecutive tokens per step with one 16-byte load and one
// 16-byte store, so a warp moves 256 tokens (512 contiguous bytes) a step.
// The three inputs before a lane's chunk are the previous lane's last three,
// passed by shuffle; lane 0 takes them from the previous step's lane 31, or
// from the initial state.  The next step's chunk is loaded while this one is
// computed, and the one after it prefetched into L2 (8% faster at 4 x 1536 x
// 2048 and at 8 x 5120 x 8192).  Same per-element operations as every other
// forward path.
template <int ACT>
__global__ void __launch_bounds__(256) fwd_bdt8_kernel(FwdArgs a) {
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_release();
  using VT = Vec<8>;
  const unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= int64_t(a.B) * a.D) return;  // the whole warp shares the row
  const int bb = int(row / a.D), d = int(row % a.D);
  float w[1][kWidth], b[1];
  load_weights_1(a.wr, d, w, b);
  const int64_t T = a.seqs.T;
  const uint16_t* xr = a.x + bb * a.x_sb + d * a.x_sd;
  uint16_t* orow = a.out + bb * a.o_sb + d * a.o_sd;
  float carry[kState];  // xe[-3 .. -1] before the row's first token
  {
    float init[kState][1] = {{0.0f}, {0.0f}, {0.0f}};
    if (a.init) load_state<1>(a.init, row, a.sw, init);
#pragma unroll
    for (int i = 0; i < kState; ++i) carry[i] = init[i][0];
  }
  typename VT::Raw nxt = make_uint4(0, 0, 0, 0);
  if (int64_t(lane) * 8 < T) nxt = VT::ld(xr + lane * 8);
  for (int64_t base = 0; base < T; base += 256) {
    const int64_t t0 = base + lane * 8;
    const bool valid = t0 < T;
    const typename VT::Raw cur = nxt;
    if (t0 + 256 < T) nxt = VT::ld(xr + t0 + 256);
    if (t0 + 512 < T) prefetch_l2(xr + t0 + 512);  // the chunk after that: into L2
    float c[8];
    VT::unpack(cur, c);
    float win[kState];
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      win[i] = __shfl_up_sync(kAll, c[8 - kState + i], 1);
      if (lane == 0) win[i] = carry[i];
    }
    float y[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float p = b[0];
      p = fmaf(w[0][0], win[0], p);
      p = fmaf(w[0][1], win[1], p);
      p = fmaf(w[0][2], win[2], p);
      p = fmaf(w[0][3], c[u], p);
      y[u] = act_fwd<ACT>(p);
      win[0] = win[1];
      win[1] = win[2];
      win[2] = c[u];
    }
    if (valid) VT::st(orow + t0, VT::pack(y));
    if (valid && t0 + 8 == T && a.fin) {  // the row's last chunk: xe[T-3 .. T-1]
      float fin[kState][1];
#pragma unroll
      for (int i = 0; i < kState; ++i) fin[i][0] = c[8 - kState + i];
      store_state<1>(a.fin, row, a.sw, fin);
    }
#pragma unroll
    for (int i = 0; i < kState; ++i) carry[i] = __shfl_sync(kAll, c[8 - kState + i], 31);
  }
}

// Time-contiguous x (stride of T is 1).  One warp per (batch, channel) row;
// lane l walks tokens [8l + 256i, 8l + 256i + 8).
template <int ACT, bool IDS = false>
__global__ void __launch_bounds__(256) fwd_bdt_kernel(FwdArgs a) {
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_release();
  if (block_rejects_cu_seqlens(a.seqs, a.status)) return;
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool dense = a.seqs.cu == nullptr;
  const int64_t rows = dense ? int64_t(a.B) * a.D : a.D;
  if (row >= rows) return;
  const int bb = int(row / a.D);
  const int d = int(row % a.D);
  float w[1][kWidth], b[1];
  load_weights_1(a.wr, d, w, b);
  // Within a row, a dense call is one sequence of T tokens (state index bb).
  Seqs rs = a.seqs;
  if (dense) { rs.Q = a.seqs.T; rs.n_seq = 1; }
  const Stream xs{bb * a.x_sb + d * a.x_sd, 0, 1};
  const Stream os{bb * a.o_sb + d * a.o_sd, 0, 1};
  for (int64_t q0 = int64_t(lane) * 8; q0 < rs.Q; q0 += 256) {
    const int64_t q1 = q0 + 8 < rs.Q ? q0 + 8 : rs.Q;
    fwd_walk<1, ACT, 4, 0, IDS>(a, rs, xs, os, dense ? bb : 0, d, w, b, q0, q1);
  }
}

// T == 0: every sequence's final state is its initial state (or zeros).
__global__ void fwd_empty_kernel(const uint16_t* init, uint16_t* fin, int64_t n) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) fin[i] = init ? init[i] : uint16_t(0);
}

// ---- host launchers ------------------------------------------------------------

// Opt the vector kernel in to its ring's dynamic shared memory (once per
// context: the attribute belongs to the module loaded in a context).
static ContextCache g_fwd_attr_done;
static cudaError_t fwd_smem_attributes() {
  long long done = 0;
  if (g_fwd_attr_done.get(&done) && done) return cudaSuccess;
  const int bytes = int(fwd_ring_bytes<4>(kFwdThreads)), bytes_ids = int(fwd_ring_bytes<4>(kFwdIdsThreads));
  cudaError_t err = cudaSuccess;
  for (auto f : {fwd_clv_kernel<4, kActSilu, true>, fwd_clv_kernel<4, kActNone, true>})
    if (err == cudaSuccess) err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes_ids);
  for (auto f : {fwd_clv_kernel<4, kActSilu>, fwd_clv_kernel<4, kActNone>,
                 fwd_clv_kernel<4, kActSilu, false, true>, fwd_clv_kernel<4, kActNone, false, true>,
                 fwd_clv_kernel<4, kActSilu, false, false, kFwdGroupShort>,
                 fwd_clv_kernel<4, kActNone, false, false, kFwdGroupShort>,
                 fwd_clv_kernel<4, kActSilu, false, true, kFwdGroupShort>,
                 fwd_clv_kernel<4, kActNone, false, true, kFwdGroupShort>})
    if (err == cudaSuccess) err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) g_fwd_attr_done.put(1);
  return err;
}

static ContextCache g_fwd_occupancy[2];
int fwd_blocks_per_sm(int vec) {
  ContextCache& cache = g_fwd_occupancy[vec == 4 ? 0 : 1];
  long long v = 0;
  if (cache.get(&v) && v > 0) return int(v);
  int n = 0;
  fwd_smem_attributes();
  const cudaError_t err =
      vec == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_clv_kernel<4, kActSilu>, kFwdThreads,
                                                               fwd_ring_bytes<4>(kFwdThreads))
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_cl_kernel<1, kActSilu>, 256, 0);
  if (err == cudaSuccess && n > 0) {
    cache.put(n);
    return n;
  }
  return 1;
}

static ContextCache g_fwd_ids_occupancy[2];
int fwd_ids_blocks_per_sm(int vec) {
  ContextCache& cache = g_fwd_ids_occupancy[vec == 4 ? 0 : 1];
  long long v = 0;
  if (cache.get(&v) && v > 0) return int(v);
  int n = 0;
  fwd_smem_attributes();
  const cudaError_t err =
      vec == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_clv_kernel<4, kActSilu, true>,
                                                               kFwdIdsThreads, fwd_ring_bytes<4>(kFwdIdsThreads))
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_cl_kernel<1, kActSilu, true>,
                                                               kGeneralThreads, 0);
  if (err == cudaSuccess && n > 0) {
    cache.put(n);
    return n;
  }
  return 1;
}

// Calls with per-token sequence ids: the ring kernel (4 channels a thread) or
// the general kernels, with id masks.
template <int ACT>
static cudaError_t launch_fwd_ids(const FwdArgs& a, const FwdPlan& p, cudaStream_t stream) {
  if (p.kind == kLayoutChannelLast) {
    dim3 block(p.tx, p.ty), grid(p.gx, p.gy);
    if (p.vec == 4) {
      const cudaError_t err = fwd_smem_attributes();
      if (err != cudaSuccess) return err;
      return launch_kernel(fwd_clv_kernel<4, ACT, true>, grid, block, fwd_ring_bytes<4>(p.tx * p.ty),
                           stream, true, a);
    }
    return launch_kernel(fwd_cl_kernel<1, ACT, true>, grid, block, 0, stream, true, a);
  }
  return launch_kernel(fwd_bdt_kernel<ACT, true>, dim3(p.gx), dim3(256), 0, stream, true, a);
}

template <int ACT>
static cudaError_t launch_fwd_act(const FwdArgs& a, const FwdPlan& p, cudaStream_t stream) {
  if (p.ids) return launch_fwd_ids<ACT>(a, p, stream);
  if (p.kind == kLayoutChannelLast) {
    dim3 block(p.tx, p.ty), grid(p.gx, p.gy);
    if (p.vec == 4) {
      const cudaError_t err = fwd_smem_attributes();
      if (err != cudaSuccess) return err;
      if (a.wr.w_vec3 && p.group == kFwdGroupShort)
        return launch_kernel(fwd_clv_kernel<4, ACT, false, true, kFwdGroupShort>, grid, block,
                             fwd_ring_bytes<4>(p.tx * p.ty, kFwdGroupShort), stream, true, a);
      if (a.wr.w_vec3)
        return launch_kernel(fwd_clv_kernel<4, ACT, false, true>, grid, block,
                             fwd_ring_bytes<4>(p.tx * p.ty), stream, true, a);
      if (p.group == kFwdGroupShort)
        return launch_kernel(fwd_clv_kernel<4, ACT, false, false, kFwdGroupShort>, grid, block,
                             fwd_ring_bytes<4>(p.tx * p.ty, kFwdGroupShort), stream, true, a);
      return launch_kernel(fwd_clv_kernel<4, ACT>, grid, block, fwd_ring_bytes<4>(p.tx * p.ty),
                           stream, true, a);
    }
    return launch_kernel(fwd_cl_kernel<1, ACT>, grid, block, 0, stream, true, a);
  }
  if (p.vec == 8) return launch_kernel(fwd_bdt8_kernel<ACT>, dim3(p.gx), dim3(256), 0, stream, true, a);
  return launch_kernel(fwd_bdt_kernel<ACT>, dim3(p.gx), dim3(256), 0, stream, true, a);
}

cudaError_t launch_fwd(const FwdArgs& a, const FwdPlan& p, int act, cudaStream_t stream) {
  if (a.seqs.Q == 0) {
    const int64_t n = int64_t(a.seqs.n_seq) * a.D * a.sw;
    if (a.fin && n > 0)
      fwd_empty_kernel<<<unsigned((n + 255) / 256), 256, 0, stream>>>(a.init, a.fin, n);
    return cudaGetLastError();
  }
  return act == kActSilu ? launch_fwd_act<kActSilu>(a, p, stream)
                         : launch_fwd_act<kActNone>(a, p, stream);
}

}  // namespace ccc
