// Backward kernels of the depthwise causal conv1d (cuDNN frontend docs, "Causal
// Conv1d" page: forward and backward on the optimized route; the paragraph on
// determinism -- FP32 atomics by default, unique FP32 partials plus a
// fixed-order reduction when deterministic).  Both modes here take the second
// route: every block writes its own row of FP32 partial sums and the finalize
// kernel adds the rows in a fixed order, so the weight gradient is always
// bitwise repeatable and no accumulator needs zeroing first.
//
// With gp[t] = dout[t] * act'(pre[t]) (pre recomputed from x, nothing saved):
//   dxe[j] = sum_k w[k] * gp[j + 3 - k]  (+ dfinal[j - (len-3)] for j >= len-3)
//   dx = dxe[0 .. len), dinit = dxe[-3 .. 0)
//   dw[k] = sum gp[t] * xe[t - 3 + k],  db = sum gp[t]
// A thread owns V channels and a token range [a, e); it walks m from a to
// e + 2, computing gp[m] (three tokens past e are recomputed, not
// accumulated) and emitting dxe[m - 3] once gp[m-3 .. m] are known.  The
// thread whose range starts a sequence also emits the three dinit entries.
// The kernels work with the halved weights and gp2 = 2 gp (see the activation
// section of common.cuh), which leaves dxe unchanged and doubles the sums,
// halved once before they are written.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace ccc {

template <int V, int ACT, int U, int P, bool IDS = false>
__device__ __forceinline__ void bwd_walk(const BwdArgs& a, const Seqs& seqs, const Stream& xs,
                                         const Stream& gs, const Stream& ds, int n_base, int d0,
                                         const float (&w)[V][kWidth], const float (&b)[V],
                                         int64_t q, int64_t q_end, float (&aw)[V][kWidth],
                                         float (&ab)[V]) {
  using VT = Vec<V>;
  int n = find_seq(seqs, q);
  while (q < q_end) {
    int64_t lo, hi;
    seq_bounds(seqs, n, lo, hi);
    const int64_t a0 = q;
    const int64_t e = q_end < hi ? q_end : hi;
    const bool starts = a0 == lo;
    const int64_t state_row = (int64_t(n_base) + n) * a.D + d0;

    float xw[kState][V];  // xe[m-3 .. m-1]
    float gw[kState][V];  // gp[m-3 .. m-1]; entries before a0 are never emitted from,
                          // except before a sequence start, where gp is zero
    float di[kState][V];  // dinit entries of this sequence (only when starts)
    // With IDS (per-token sequence ids, cuDNN page seq_idx[B, T]): iw = ids of
    // tokens m-3 .. m-1 (any value before the row start, where x and gp are
    // zero); token t's id is at id_off + t * ids_st.  A tap joins two tokens
    // only when their ids are equal.
    int iw[kState] = {0, 0, 0};
    const int64_t id_off = IDS ? (int64_t(n_base) + n) * a.ids_sb - lo * a.ids_st : 0;
    {
      float init[kState][V];
      if (a0 - kState < lo && a.init) {
        load_state<V>(a.init, state_row, a.sw, init);
      } else {
#pragma unroll
        for (int i = 0; i < kState; ++i)
#pragma unroll
          for (int c = 0; c < V; ++c) init[i][c] = 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kState; ++j) {
        const int64_t tok = a0 - kState + j;
        if (tok >= lo) {
          VT::unpack(VT::ld(a.x + xs.at(n, tok)), xw[j]);
          if constexpr (IDS) iw[j] = __ldg(a.ids + id_off + tok * a.ids_st);
        } else {
          const int64_t i = tok - lo + kState;
#pragma unroll
          for (int c = 0; c < V; ++c)
            xw[j][c] = i == 0 ? init[0][c] : (i == 1 ? init[1][c] : init[2][c]);
        }
#pragma unroll
        for (int c = 0; c < V; ++c) { gw[j][c] = 0.0f; di[j][c] = 0.0f; }
      }
    }
    // id of token m (IDS), read once per step by grad_at and emit
    int cid = 0;

    // gp at token m from its inputs; accumulate the weight/bias sums when m is
    // one of this thread's tokens; shift the input window.
    auto grad_at = [&](typename VT::Raw xr, typename VT::Raw gr, bool own, float (&gp)[V]) {
      float xc[V], gc[V];
      VT::unpack(xr, xc);
      VT::unpack(gr, gc);
      bool m0 = true, m1 = true, m2 = true;  // window token k feeds token m
      if constexpr (IDS) {
        m0 = iw[0] == cid;
        m1 = iw[1] == cid;
        m2 = iw[2] == cid;
      }
#pragma unroll
      for (int c = 0; c < V; ++c) {
        const float x0 = m0 ? xw[0][c] : 0.0f, x1 = m1 ? xw[1][c] : 0.0f,
                    x2 = m2 ? xw[2][c] : 0.0f;
        float p = b[c];
        p = fmaf(w[c][0], x0, p);
        p = fmaf(w[c][1], x1, p);
        p = fmaf(w[c][2], x2, p);
        p = fmaf(w[c][3], xc[c], p);
        gp[c] = act_bwd<ACT>(p, gc[c]);
        if (own) {
          aw[c][0] = fmaf(gp[c], x0, aw[c][0]);
          aw[c][1] = fmaf(gp[c], x1, aw[c][1]);
          aw[c][2] = fmaf(gp[c], x2, aw[c][2]);
          aw[c][3] = fmaf(gp[c], xc[c], aw[c][3]);
          ab[c] += gp[c];
        }
        xw[0][c] = xw[1][c];
        xw[1][c] = xw[2][c];
        xw[2][c] = xc[c];
      }
    };
    // dxe[m - 3] from gp[m] and the window gp[m-3 .. m-1]; shift the windows.
    auto emit = [&](const float (&gp)[V], float (&v)[V]) {
      bool e2 = true, e1 = true, e0 = true;  // token m-3 feeds the tap of token m-2, m-1, m
      if constexpr (IDS) {
        e2 = iw[0] == iw[1];
        e1 = iw[0] == iw[2];
        e0 = iw[0] == cid;
        iw[0] = iw[1];
        iw[1] = iw[2];
        iw[2] = cid;
      }
#pragma unroll
      for (int c = 0; c < V; ++c) {
        float s = w[c][3] * gw[0][c];  // oldest first: gp[m] enters last
        s = fmaf(w[c][2], e2 ? gw[1][c] : 0.0f, s);
        s = fmaf(w[c][1], e1 ? gw[2][c] : 0.0f, s);
        s = fmaf(w[c][0], e0 ? gp[c] : 0.0f, s);
        v[c] = s;
        gw[0][c] = gw[1][c];
        gw[1][c] = gw[2][c];
        gw[2][c] = gp[c];
      }
    };

    // General step: any m in [a0, e + 3).
    auto slow = [&](int64_t m) {
      float gp[V], v[V];
      if (m < hi) {
        if constexpr (IDS) cid = __ldg(a.ids + id_off + m * a.ids_st);
        grad_at(VT::ld(a.x + xs.at(n, m)), VT::ld(a.g + gs.at(n, m)), m < e, gp);
      } else {
#pragma unroll
        for (int c = 0; c < V; ++c) gp[c] = 0.0f;
      }
      const int64_t j = m - kState;
      emit(gp, v);
      if (j >= a0 || starts) {
        if (a.dfin && j >= hi - kState) {
          const int i = int(j - (hi - kState));  // window slot of the final state
#pragma unroll
          for (int c = 0; c < V; ++c) {
            const int64_t k = state_slot(state_row + c, i, a.sw);
            if (k >= 0) v[c] += bf16_to_f32(__ldg(a.dfin + k));
          }
        }
        if (j >= lo) {
          VT::st(a.dx + ds.at(n, j), VT::pack(v));
        } else if (a.dinit) {
          const int64_t i = j - lo + kState;
#pragma unroll
          for (int c = 0; c < V; ++c) {
            if (i == 0) di[0][c] = v[c];
            else if (i == 1) di[1][c] = v[c];
            else di[2][c] = v[c];
          }
          if (i == kState - 1) store_state<V>(a.dinit, state_row, a.sw, di);
        }
      }
    };

    int64_t m = a0;
    const int64_t m_end = e + kState;
    const int64_t pro_end = a0 + kState < m_end ? a0 + kState : m_end;
    // rows this piece reads: [a0, min(e + 3, hi)); prefetch P rows ahead into L2
    const int64_t r_end = m_end < hi ? m_end : hi;
    if constexpr (P > 0) {
      for (int64_t t = a0 + kState; t < a0 + kState + P && t < r_end; ++t) {
        prefetch_l2(a.x + xs.at(n, t));
        prefetch_l2(a.g + gs.at(n, t));
      }
    }
    for (; m < pro_end; ++m) slow(m);
    // steady state: own tokens, emissions land in [a0, e - 3), no state involved
    for (; m + U <= e; m += U) {
      if constexpr (P > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t t = m + P + u;
          if (t < r_end) {
            prefetch_l2(a.x + xs.at(n, t));
            prefetch_l2(a.g + gs.at(n, t));
          }
        }
      }
      typename VT::Raw xr[U], gr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        xr[u] = VT::ld(a.x + xs.at(n, m + u));
        gr[u] = VT::ld(a.g + gs.at(n, m + u));
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float gp[V], v[V];
        if constexpr (IDS) cid = __ldg(a.ids + id_off + (m + u) * a.ids_st);
        grad_at(xr[u], gr[u], true, gp);
        emit(gp, v);
        VT::st(a.dx + ds.at(n, m + u - kState), VT::pack(v));
      }
    }
    for (; m < m_end; ++m) slow(m);

    q = e;
    ++n;
  }
}

// Dynamic shared memory of the channel-last backward kernels: the block's
// weight/bias sums for the final reduction ([ty][tx][V * 5] floats), then (the
// vector kernels) each thread's ring of staged input rows.
extern __shared__ __align__(16) float bwd_dyn_smem[];
template <int V>
__host__ __device__ constexpr size_t bwd_red_bytes(int threads) {
  return size_t(threads) * V * (kWidth + 1) * sizeof(float);
}

// Block-wide sum of the per-thread weight/bias sums (sums of gp2 = 2 gp, halved
// here) over threadIdx.y (threads with equal threadIdx.x own the same
// channels), in a fixed order, stored into this block row's own partial row
// ws[blockIdx.y].  No atomics: every value of the row is written, so the
// workspace needs no zeroing and its contents on entry are never read.
template <int V>
__device__ __forceinline__ void block_wgrad_out(const BwdArgs& a, int d0, bool active,
                                                const float (&aw)[V][kWidth], const float (&ab)[V]) {
  float* red = bwd_dyn_smem;  // [ty][tx][V * 5]
  constexpr int P = V * (kWidth + 1);
  float* mine = red + (threadIdx.y * blockDim.x + threadIdx.x) * P;
#pragma unroll
  for (int c = 0; c < V; ++c) {
#pragma unroll
    for (int k = 0; k < kWidth; ++k) mine[c * (kWidth + 1) + k] = active ? 0.5f * aw[c][k] : 0.0f;
    mine[c * (kWidth + 1) + kWidth] = active ? 0.5f * ab[c] : 0.0f;
  }
  __syncthreads();
  // each of the block's threads finalises a slice of the tx * P values
  const int nthr = blockDim.x * blockDim.y;
  const int tid = threadIdx.y * blockDim.x + threadIdx.x;
  const int total = blockDim.x * P;
  const int dbase = blockIdx.x * blockDim.x * V;
  for (int i = tid; i < total; i += nthr) {
    const int tx = i / P, r = i % P;
    const int d = dbase + tx * V + r / (kWidth + 1);
    if (d >= a.D) continue;
    float s = 0.0f;
    for (int y = 0; y < int(blockDim.y); ++y) s += red[(y * blockDim.x + tx) * P + r];
    const int k = r % (kWidth + 1);
    a.ws[(int64_t(blockIdx.y) * a.D + d) * (kWidth + 1) + k] = s;
  }
}

template <int V, int ACT, bool IDS = false>
__global__ void __launch_bounds__(kGeneralThreads) bwd_cl_kernel(BwdArgs a) {
  __shared__ __align__(16) float wsm[(kWidth + 1) * kMaxBlockChannels];
  pdl_wait();  // inputs may come from the previous kernel in the stream
  if (block_rejects_cu_seqlens(a.seqs, a.status)) return;
  const int n_blk = blockDim.x * V;
  stage_weights(a.wr, blockIdx.x * n_blk, n_blk, a.D, wsm);
  const int d0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
  const int64_t seg = int64_t(blockIdx.y) * blockDim.y + threadIdx.y;
  const bool active = d0 < a.D && seg < a.n_seg;
  float aw[V][kWidth], ab[V];
#pragma unroll
  for (int c = 0; c < V; ++c) {
    ab[c] = 0.0f;
#pragma unroll
    for (int k = 0; k < kWidth; ++k) aw[c][k] = 0.0f;
  }
  if (active) {
    float w[V][kWidth], b[V];
    weights_from_smem<V>(wsm, n_blk, threadIdx.x * V, w, b);
    int64_t q0, q1;
    seg_range(a.seqs, seg, a.seg_len, a.seg_per_seq, q0, q1);
    const bool dense = a.seqs.cu == nullptr;
    const Stream xs{d0, dense ? a.x_sb - a.seqs.T * a.x_st : 0, a.x_st};
    const Stream gs{d0, dense ? a.g_sb - a.seqs.T * a.g_st : 0, a.g_st};
    const Stream ds{d0, dense ? a.dx_sb - a.seqs.T * a.dx_st : 0, a.dx_st};
    bwd_walk<V, ACT, 4, (V == 8 ? 16 : 0), IDS>(a, a.seqs, xs, gs, ds, 0, d0, w, b, q0, q1, aw, ab);
  }
  pdl_release();
  block_wgrad_out<V>(a, d0, active, aw, ab);
}

// Channel-last backward with vectors of V = 8 or 4 channels (the fast path).
// Same walk as bwd_walk, specialised like fwd_clv_kernel: the input window and
// the gradient window rotate through three register slots and the own tokens
// of a piece are taken in groups of three.  Those groups' rows (x and
// grad_out) stream through the thread's own ring of kBwdRing stages in shared
// memory with cp.async, kBwdRing - 1 groups ahead of the group being computed,
// so the steady loop never waits on a load it has just issued and holds no
// registers for loads in flight.  The ring's first group is the head (own
// tokens whose dx rows belong to the previous piece) and its last the tail
// (the three tokens after the piece, which emit its last dx rows); the few
// tokens at sequence edges take the general step, loading their rows directly
// (prefetched into L2 when the piece starts).
// 256-thread blocks: one resident per SM for V = 8, two for V = 4 (the id
// instance: one 384-thread block per SM).
#ifndef CCC_BWD_RING
#define CCC_BWD_RING 3
#endif
constexpr int kBwdRing = CCC_BWD_RING;
static_assert(kBwdRing >= 2, "the ring needs a stage being filled and one being read");
template <int V>
constexpr size_t bwd_ring_bytes(int threads) {
  return size_t(threads) * kBwdRing * 3 * 2 * (2 * V);
}
// Threads a block: 256 for eight channels a thread (one block an SM, ~240
// registers) and for four (two blocks an SM, 128 registers); 384 for the id
// instance (~150 registers, one block an SM: 27.3 us with seq_idx at
// 4 x 2048 x 1536 against 27.6 us for three 128-thread blocks and 29.0 us for
// two of 192).  Measured: at eight channels,
// 256-thread blocks took 307 us against 311 us at 8 x 5120 x 8192 and 78.8
// against 80.5 us on 16 packed sequences (half the partial rows).  At four,
// with segments planned per sequence, 4 x 2048 x 1536 took 20.9-21.1 us in
// 256-thread blocks against 21.7-21.8 us in 128 and 21.5 us in 512: the warp
// scheduler favours a block's older warps, so with four blocks an SM the
// last-placed block ran its loop about 4 us behind the first and finished
// with the SM mostly idle.
#ifndef CCC_BWD_IDS_THREADS
#define CCC_BWD_IDS_THREADS 384
#endif
template <int V, bool IDS = false>
__host__ __device__ constexpr int bwd_threads() { return V == 8 || !IDS ? 256 : CCC_BWD_IDS_THREADS; }

// With IDS (V = 4; dense calls without states), every token carries a sequence
// id (cuDNN page, seq_idx[B, T]): a tap joins two tokens only when their ids
// are equal.  A ring group whose three tokens and the three before them share
// one id (all but the groups at an id change, for ids that form runs) takes
// the fast steps; any other takes the general step, which masks every tap by
// the ids.  Both leave the windows at phase 0 after a group.
#ifndef CCC_BWD_IDS_BLOCKS
#define CCC_BWD_IDS_BLOCKS 1  // resident blocks an SM asked of the id instance
#endif
template <int V, int ACT, bool IDS = false>
__global__ void __launch_bounds__(bwd_threads<V, IDS>(), V == 8 ? 1 : (IDS ? CCC_BWD_IDS_BLOCKS : 2))
    bwd_clv_kernel(BwdArgs a) {
  using VT = Vec<V>;
  using Raw = typename VT::Raw;
  constexpr int H = V / 2;  // channel pairs
  constexpr int RB = int(sizeof(Raw));
  __shared__ __align__(16) float wsm[(kWidth + 1) * (V == 8 ? 2 * kMaxBlockChannels : kMaxBlockChannels)];
  constexpr int NT = bwd_threads<V, IDS>();
  if (blockDim.x * blockDim.y * blockDim.z != NT) return;  // the ring layout assumes it
  pdl_wait();  // inputs may come from the previous kernel in the stream
  if (block_rejects_cu_seqlens(a.seqs, a.status)) return;
  const int n_blk = blockDim.x * V;
  const int d0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
  const int64_t seg = int64_t(blockIdx.y) * blockDim.y + threadIdx.y;
  const bool active = d0 < a.D && seg < a.n_seg;
  if (!a.wr.w_vec && !a.wr.w_vec3) stage_weights(a.wr, blockIdx.x * n_blk, n_blk, a.D, wsm);  // block-uniform
  float2 aw[H][kWidth], ab[H];
#pragma unroll
  for (int h = 0; h < H; ++h) {
    ab[h] = splat2(0.0f);
#pragma unroll
    for (int k = 0; k < kWidth; ++k) aw[h][k] = splat2(0.0f);
  }
  if (active) {
    float2 w[H][kWidth], b[H];
    bool have_w = false;  // the weights are loaded once the first ring groups are in flight
    // this thread's ring: slot (stage, row u, tensor t) at byte
    // (((stage * 3 + u) * 2 + t) * NT + tid) * RB past the ring base: the
    // block size is a compile-time constant, so every offset is an immediate
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    const char* ring = reinterpret_cast<const char*>(bwd_dyn_smem) + bwd_red_bytes<V>(NT) +
                       size_t(tid) * RB;
    const uint32_t ring_s = smem_u32(ring);
    constexpr uint32_t slot = uint32_t(NT) * RB;

    int64_t q, q_end;
    seg_range(a.seqs, seg, a.seg_len, a.seg_per_seq, q, q_end);
    const bool dense = a.seqs.cu == nullptr;
    int n = find_seq(a.seqs, q);
    using P0 = std::integral_constant<int, 0>;
    using P1 = std::integral_constant<int, 1>;
    using P2 = std::integral_constant<int, 2>;
    using Yes = std::true_type;
    using No = std::false_type;
    while (q < q_end) {
      int64_t lo, hi;
      seq_bounds(a.seqs, n, lo, hi);
      const int64_t a0 = q;
      const int64_t e = q_end < hi ? q_end : hi;
      const bool starts = a0 == lo;
      const int64_t state_row = int64_t(n) * a.D + d0;
      const int64_t xst = a.x_st, gst = a.g_st, dst = a.dx_st;
      // IW: ids of tokens m-3 .. m-1 (IDS; any value before the row start,
      // where x and gp are zero); token t's id is at id_off + t * ids_st
      int IW[kState] = {0, 0, 0};
      const int64_t id_off = IDS ? int64_t(n) * a.ids_sb - lo * a.ids_st : 0;
      auto id_at = [&](int64_t t) { return __ldg(a.ids + id_off + t * a.ids_st); };
      // pointers at token a0
      const uint16_t* xp = a.x + (dense ? n * a.x_sb + (a0 - lo) * xst : a0 * xst) + d0;
      const uint16_t* gq = a.g + (dense ? n * a.g_sb + (a0 - lo) * gst : a0 * gst) + d0;
      uint16_t* dp = a.dx + (dense ? n * a.dx_sb + (a0 - lo) * dst : a0 * dst) + d0;
      const int64_t m_end = e + kState;  // tokens stepped: [a0, e + 3)
      // The ring's groups: rows r0 + 3k .. r0 + 3k + 2 for k < n_total.  With a
      // head (the window came from x rows and a0 .. a0+2 are own) r0 = a0 and
      // group 0 computes own tokens whose emissions are the previous piece's
      // rows; otherwise the first three tokens take the general step and
      // r0 = a0 + 3.  Then the groups of own tokens emitting own rows; then,
      // when those end on e with three more rows in the sequence, the tail
      // group, which emits the last own rows; else the general step finishes.
      // The first groups go out before anything else of the piece is read but
      // the window (halo rows or initial state) and the weights.
      const bool head = a0 - kState >= lo && a0 + 3 <= e;
      // A sequence's first piece, when it holds three tokens and the sequence
      // six: its first ring group takes those tokens too, with the window from
      // the initial state, and the group's emissions become the initial
      // state's gradient (the general step's arithmetic, in its order).
      const bool shead = !IDS && starts && a0 + 3 <= e && hi - lo >= 2 * kState;
      const int64_t r0 = head || shead ? a0 : (a0 + kState < m_end ? a0 + kState : m_end);
      const int n_main = e > r0 ? int((e - r0) / 3) : 0;  // a segment's groups: below 2^31
      const bool tail = e > r0 && (e - r0) % 3 == 0 && e + kState <= hi && e - a0 >= kState;
      const int n_total = n_main + (tail ? 1 : 0);
      // running pointers: the next group to issue (rows and ring stage), the
      // group being taken (stage, dx rows)
      const uint16_t* xi = xp + (r0 - a0) * xst;
      const uint16_t* gi = gq + (r0 - a0) * gst;
      int ki = 0, si = 0;  // next group to issue, its stage
      auto issue_next = [&]() {
        if (ki < n_total) {
          const uint32_t s0 = ring_s + uint32_t(si * 6) * slot;
#pragma unroll
          for (int u = 0; u < 3; ++u) {
            cp_async<RB>(s0 + uint32_t(2 * u) * slot, xi + u * xst);
            cp_async<RB>(s0 + uint32_t(2 * u + 1) * slot, gi + u * gst);
          }
          xi += 3 * xst;
          gi += 3 * gst;
        }
        ++ki;
        si = (si + 1) % kBwdRing;
        cp_async_commit();
      };
      int st = 0;  // stage of the group being taken
      // takes the group of tokens m0 .. m0 + 2; true when they and the three
      // tokens before them share one id (always without IDS)
      auto take = [&](Raw (&xr)[3], Raw (&gr)[3], int64_t m0) {
        issue_next();
        bool uniform = true;
        if constexpr (IDS) {
          uniform = IW[0] == IW[1] && IW[1] == IW[2];
#pragma unroll
          for (int u = 0; u < 3; ++u) uniform = uniform && id_at(m0 + u) == IW[2];
        }
        cp_async_wait<kBwdRing - 1>();  // the group being taken has landed
        const char* s0 = ring + size_t(st * 6) * slot;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          xr[u] = *reinterpret_cast<const Raw*>(s0 + size_t(2 * u) * slot);
          gr[u] = *reinterpret_cast<const Raw*>(s0 + size_t(2 * u + 1) * slot);
        }
        st = (st + 1) % kBwdRing;
        return uniform;
      };
      // The window's own loads (the halo rows, or the initial state) and the
      // weights go out before the ring's first groups: the first step needs
      // all of them, and requests are served about in the order issued.
      // Measured: 4 x 2048 x 1536 20.85 -> 20.07 us, with seq_idx 27.4 ->
      // 26.4 us; 16 packed sequences 77.86 -> 77.25 us; 8 x 5120 x 8192
      // 302.8 -> 301.9 us.
      float2 X[kState][H], G[kState][H];  // xe[m-3 .. m-1], gp[m-3 .. m-1]
      if constexpr (IDS) {
#pragma unroll
        for (int j = 0; j < kState; ++j)
          if (a0 - kState + j >= lo) IW[j] = id_at(a0 - kState + j);
      }
      {
        float2 init[kState][H];
        if (a0 - kState < lo && a.init) {
          load_state2<V>(a.init, state_row, a.sw, init);
        } else {
#pragma unroll
          for (int i = 0; i < kState; ++i)
#pragma unroll
            for (int h = 0; h < H; ++h) init[i][h] = splat2(0.0f);
        }
        Raw hx[kState] = {};  // halo rows, unpacked once the ring's first groups are out
#pragma unroll
        for (int j = 0; j < kState; ++j)
          if (a0 - kState + j >= lo) hx[j] = VT::ld(xp - (kState - j) * xst);
        if (!have_w) {
          if (a.wr.w_vec || a.wr.w_vec3) weights_direct2_any<V>(a.wr, d0, w, b);
          else weights_from_smem2<V>(wsm, n_blk, threadIdx.x * V, w, b);
          have_w = true;
        }
#pragma unroll
        for (int j = 0; j < kBwdRing - 1; ++j) issue_next();
        // rows the general steps may read at the piece's two ends: into L2
        const int64_t r_end = m_end < hi ? m_end : hi;
        for (int64_t t = a0; t < a0 + kState && t < r_end; ++t) {
          prefetch_l2(xp + (t - a0) * xst);
          prefetch_l2(gq + (t - a0) * gst);
        }
        for (int64_t t = (e - 2 > a0 + kState ? e - 2 : a0 + kState); t < r_end; ++t) {
          prefetch_l2(xp + (t - a0) * xst);
          prefetch_l2(gq + (t - a0) * gst);
        }
        // X[j] from halo row j or the initial state; G zero
#pragma unroll
        for (int j = 0; j < kState; ++j) {
          const int64_t tok = a0 - kState + j;
          if (tok >= lo) {
            VT::unpack2(hx[j], X[j]);
          } else {
            const int64_t i = tok - lo + kState;
#pragma unroll
            for (int h = 0; h < H; ++h)
              X[j][h] = i == 0 ? init[0][h] : (i == 1 ? init[1][h] : init[2][h]);
          }
#pragma unroll
          for (int h = 0; h < H; ++h) G[j][h] = splat2(0.0f);
        }
      }

      // general step at token m, windows at phase 0 (physical shifts)
      auto slow = [&](int64_t m) {
        float2 gp[H], v[H];
        // IDS: the forward taps read window token k only when its id is token
        // m's (f0..f2); dx[m-3] takes gp of m-2, m-1, m only when their ids are
        // token m-3's (e1, e2, e3)
        int cid = 0;
        bool f0 = true, f1 = true, f2 = true, e1 = true, e2 = true, e3 = true;
        if constexpr (IDS) {
          if (m < hi) cid = id_at(m);
          f0 = IW[0] == cid;
          f1 = IW[1] == cid;
          f2 = IW[2] == cid;
          e1 = IW[1] == IW[0];
          e2 = IW[2] == IW[0];
          e3 = cid == IW[0];
          IW[0] = IW[1];
          IW[1] = IW[2];
          IW[2] = cid;
        }
        const float2 zero2 = splat2(0.0f);
        if (m < hi) {
          float2 xc[H], gc[H];
          VT::unpack2(VT::ld(xp + (m - a0) * xst), xc);
          VT::unpack2(VT::ld(gq + (m - a0) * gst), gc);
          const bool own = m < e;
#pragma unroll
          for (int h = 0; h < H; ++h) {
            const float2 x0 = f0 ? X[0][h] : zero2, x1 = f1 ? X[1][h] : zero2,
                         x2 = f2 ? X[2][h] : zero2;
            float2 p = b[h];
            p = ffma2(w[h][0], x0, p);
            p = ffma2(w[h][1], x1, p);
            p = ffma2(w[h][2], x2, p);
            p = ffma2(w[h][3], xc[h], p);
            gp[h] = act_bwd2<ACT>(p, gc[h]);
            if (own) {
              aw[h][0] = ffma2(gp[h], x0, aw[h][0]);
              aw[h][1] = ffma2(gp[h], x1, aw[h][1]);
              aw[h][2] = ffma2(gp[h], x2, aw[h][2]);
              aw[h][3] = ffma2(gp[h], xc[h], aw[h][3]);
              ab[h] = fadd2(ab[h], gp[h]);
            }
            X[0][h] = X[1][h];
            X[1][h] = X[2][h];
            X[2][h] = xc[h];
          }
        } else {
#pragma unroll
          for (int h = 0; h < H; ++h) gp[h] = zero2;
        }
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float2 acc = fmul2(w[h][3], G[0][h]);
          acc = ffma2(w[h][2], e1 ? G[1][h] : zero2, acc);
          acc = ffma2(w[h][1], e2 ? G[2][h] : zero2, acc);
          acc = ffma2(w[h][0], e3 ? gp[h] : zero2, acc);
          v[h] = acc;
          G[0][h] = G[1][h];
          G[1][h] = G[2][h];
          G[2][h] = gp[h];
        }
        const int64_t j = m - kState;
        if (j >= a0 || starts) {
          if (a.dfin && j >= hi - kState) {
            const int i = int(j - (hi - kState));  // window slot of the final state
#pragma unroll
            for (int h = 0; h < H; ++h) {
              const int64_t k0 = state_slot(state_row + 2 * h, i, a.sw);
              const int64_t k1 = state_slot(state_row + 2 * h + 1, i, a.sw);
              if (k0 >= 0) v[h].x += bf16_to_f32(__ldg(a.dfin + k0));
              if (k1 >= 0) v[h].y += bf16_to_f32(__ldg(a.dfin + k1));
            }
          }
          if (j >= lo) {
            VT::st(dp + (j - a0) * dst, VT::pack2(v));
          } else if (a.dinit) {  // one of the three entries before the sequence
            const int i = int(j - lo + kState);
#pragma unroll
            for (int h = 0; h < H; ++h) {
              const int64_t k0 = state_slot(state_row + 2 * h, i, a.sw);
              const int64_t k1 = state_slot(state_row + 2 * h + 1, i, a.sw);
              if (k0 >= 0) a.dinit[k0] = f32_to_bf16(v[h].x);
              if (k1 >= 0) a.dinit[k1] = f32_to_bf16(v[h].y);
            }
          }
        }
      };

      // steady step at window phase J for token m: with ACC, m is an own token
      // (weight/bias sums); with STORE, the emission dx[m-3] is an own row.
      auto fast = [&](auto phase, auto acc_flag, auto store_flag, Raw xr, Raw gr, uint16_t* drow) {
        constexpr int J = decltype(phase)::value;
        constexpr bool ACC = decltype(acc_flag)::value, STORE = decltype(store_flag)::value;
        constexpr int J1 = (J + 1) % 3, J2 = (J + 2) % 3;
        float2 xc[H], gc[H], v[H];
        VT::unpack2(xr, xc);
        VT::unpack2(gr, gc);
#pragma unroll
        for (int h = 0; h < H; ++h) {
          float2 p = b[h];
          p = ffma2(w[h][0], X[J][h], p);
          p = ffma2(w[h][1], X[J1][h], p);
          p = ffma2(w[h][2], X[J2][h], p);
          p = ffma2(w[h][3], xc[h], p);
          const float2 gp = act_bwd2<ACT>(p, gc[h]);
          if constexpr (ACC) {
            aw[h][0] = ffma2(gp, X[J][h], aw[h][0]);
            aw[h][1] = ffma2(gp, X[J1][h], aw[h][1]);
            aw[h][2] = ffma2(gp, X[J2][h], aw[h][2]);
            aw[h][3] = ffma2(gp, xc[h], aw[h][3]);
            ab[h] = fadd2(ab[h], gp);
          }
          X[J][h] = xc[h];
          float2 acc = fmul2(w[h][3], G[J][h]);  // independent of this token's gp
          acc = ffma2(w[h][2], G[J1][h], acc);
          acc = ffma2(w[h][1], G[J2][h], acc);
          acc = ffma2(w[h][0], gp, acc);
          v[h] = acc;
          G[J][h] = gp;
        }
        if constexpr (STORE) VT::st(drow, VT::pack2(v));
      };
      auto group = [&](auto acc_flag, auto store_flag, const Raw (&xr)[3], const Raw (&gr)[3],
                       uint16_t* drow) {
        fast(P0{}, acc_flag, store_flag, xr[0], gr[0], drow);
        fast(P1{}, acc_flag, store_flag, xr[1], gr[1], drow + dst);
        fast(P2{}, acc_flag, store_flag, xr[2], gr[2], drow + 2 * dst);
      };

      int64_t m = a0;  // general steps before the ring's first group
      if (!head) {
        for (; m < r0; ++m) slow(m);
      }
      Raw xr[3], gr[3];
      int k = 0;
      // dx rows of group k (a first group that stores nothing gets dp)
      uint16_t* drow = shead ? dp : dp + (r0 - kState - a0) * dst;
      // a group of other ids than its window's takes the general steps
      auto mixed = [&](int64_t m0) {
#pragma unroll 1
        for (int u = 0; u < 3; ++u) slow(m0 + u);
      };
      if (head) {
        if (take(xr, gr, r0)) group(Yes{}, No{}, xr, gr, drow);
        else mixed(r0);
        k = 1;
        drow += 3 * dst;
      } else if (shead) {
        take(xr, gr, r0);  // no ids: always uniform
        group(Yes{}, No{}, xr, gr, drow);
        // G[u] now holds gp of token lo + u.  Entry i of the initial state
        // (token lo - 3 + i) is the emission at token lo + i, whose taps on
        // tokens before lo read zero; no final-state gradient reaches it.
        if (a.dinit) {
          const float2 zero2 = splat2(0.0f);
#pragma unroll
          for (int i = 0; i < kState; ++i) {
#pragma unroll
            for (int h = 0; h < H; ++h) {
              const float2 gm2 = i == 2 ? G[0][h] : zero2;  // gp of token lo + i - 2
              const float2 gm1 = i == 2 ? G[1][h] : (i == 1 ? G[0][h] : zero2);
              float2 acc = fmul2(w[h][3], zero2);
              acc = ffma2(w[h][2], gm2, acc);
              acc = ffma2(w[h][1], gm1, acc);
              acc = ffma2(w[h][0], G[i][h], acc);
              const int64_t k0 = state_slot(state_row + 2 * h, i, a.sw);
              const int64_t k1 = state_slot(state_row + 2 * h + 1, i, a.sw);
              if (k0 >= 0) a.dinit[k0] = f32_to_bf16(acc.x);
              if (k1 >= 0) a.dinit[k1] = f32_to_bf16(acc.y);
            }
          }
        }
        k = 1;  // drow stays at dp: group 1 emits rows lo .. lo + 2
      }
      for (; k < n_main; ++k) {
        const int64_t m0 = r0 + 3 * int64_t(k);
        if (take(xr, gr, m0)) group(Yes{}, Yes{}, xr, gr, drow);
        else mixed(m0);
        drow += 3 * dst;
      }
      m = r0 + 3 * int64_t(n_main);
      if (tail) {
        if (take(xr, gr, m)) group(No{}, Yes{}, xr, gr, drow);
        else mixed(m);
      } else {
        for (; m < m_end; ++m) slow(m);
      }

      q = e;
      ++n;
    }
  }
  float awf[V][kWidth], abf[V];
#pragma unroll
  for (int h = 0; h < H; ++h) {
#pragma unroll
    for (int k = 0; k < kWidth; ++k) { awf[2 * h][k] = aw[h][k].x; awf[2 * h + 1][k] = aw[h][k].y; }
    abf[2 * h] = ab[h].x;
    abf[2 * h + 1] = ab[h].y;
  }
  pdl_release();  // the finalize kernel may start launching
  block_wgrad_out<V>(a, d0, active, awf, abf);
}

// Time-contiguous layout: one warp per (batch, channel) row, lane l walks
// tokens [8l + 256i, 8l + 256i + 8).  The row's sums are reduced across the
// warp in a fixed butterfly order; partial row = batch index.
template <int ACT, bool IDS = false>
__global__ void __launch_bounds__(256) bwd_bdt_kernel(BwdArgs a) {
  pdl_wait();  // inputs may come from the previous kernel in the stream
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
  Seqs rs = a.seqs;
  if (dense) { rs.Q = a.seqs.T; rs.n_seq = 1; }
  const Stream xs{bb * a.x_sb + d * a.x_sd, 0, 1};
  const Stream gs{bb * a.g_sb + d * a.g_sd, 0, 1};
  const Stream ds{bb * a.dx_sb + d * a.dx_sd, 0, 1};
  float aw[1][kWidth] = {{0.0f, 0.0f, 0.0f, 0.0f}}, ab[1] = {0.0f};
  for (int64_t q0 = int64_t(lane) * 8; q0 < rs.Q; q0 += 256) {
    const int64_t q1 = q0 + 8 < rs.Q ? q0 + 8 : rs.Q;
    bwd_walk<1, ACT, 4, 0, IDS>(a, rs, xs, gs, ds, dense ? bb : 0, d, w, b, q0, q1, aw, ab);
  }
  pdl_release();
  // the sums are of gp2 = 2 gp: halve them (exact)
  float v[kWidth + 1] = {0.5f * aw[0][0], 0.5f * aw[0][1], 0.5f * aw[0][2], 0.5f * aw[0][3],
                         0.5f * ab[0]};
#pragma unroll
  for (int k = 0; k < kWidth + 1; ++k)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], off);
  if (lane == 0) {
    for (int k = 0; k < kWidth + 1; ++k)
      a.ws[(int64_t(dense ? bb : 0) * a.D + d) * (kWidth + 1) + k] = v[k];
  }
}

// Time-contiguous, dense, T a multiple of 8 and 16-byte aligned rows: one warp
// per (batch, channel) row, each lane 8 consecutive tokens per step (16-byte
// loads of x and grad_out, 16-byte stores of dx), a warp step 256 tokens.  The
// steps are software-pipelined by one: step s computes gp2 (and the weight
// sums) of chunk s + 1 and emits the dx rows of chunk s, whose last three need
// gp2 of the three tokens after the chunk -- the next lane's first three of
// chunk s (shuffled down), or for lane 31 lane 0's of chunk s + 1.  The inputs
// before a chunk come from the previous lane (lane 0: lane 31 of the previous
// chunk, or the initial state).  Every gp2 is computed once.  The row's sums
// are reduced across the warp in a fixed butterfly order; partial row = batch
// index.
template <int ACT>
__global__ void __launch_bounds__(256) bwd_bdt8_kernel(BwdArgs a) {
  pdl_wait();  // inputs may come from the previous kernel in the stream
  using VT = Vec<8>;
  const unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= int64_t(a.B) * a.D) return;  // the whole warp shares the row
  const int bb = int(row / a.D), d = int(row % a.D);
  float w[1][kWidth], b[1];
  load_weights_1(a.wr, d, w, b);
  const float w0 = w[0][0], w1 = w[0][1], w2 = w[0][2], w3 = w[0][3];
  const int64_t T = a.seqs.T;
  const uint16_t* xr = a.x + bb * a.x_sb + d * a.x_sd;
  const uint16_t* gr = a.g + bb * a.g_sb + d * a.g_sd;
  uint16_t* dxr = a.dx + bb * a.dx_sb + d * a.dx_sd;
  float carry[kState];  // for lane 0: xe of the three tokens before its next chunk
  {
    float init[kState][1] = {{0.0f}, {0.0f}, {0.0f}};
    if (a.init) load_state<1>(a.init, row, a.sw, init);
#pragma unroll
    for (int i = 0; i < kState; ++i) carry[i] = init[i][0];
  }
  float aw[kWidth] = {0.0f, 0.0f, 0.0f, 0.0f}, ab = 0.0f;

  // gp2 of the chunk at t0 (zero for t0 >= T); accumulates the weight sums
  auto chunk_gp = [&](int64_t t0, typename VT::Raw xraw, typename VT::Raw graw, float (&gp)[8]) {
    float xe[11], gv[8];
    {
      float cx[8];
      VT::unpack(xraw, cx);
      VT::unpack(graw, gv);
#pragma unroll
      for (int u = 0; u < 8; ++u) xe[3 + u] = cx[u];
    }
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      const float px = __shfl_up_sync(kAll, xe[3 + 8 - kState + i], 1);
      xe[i] = lane == 0 ? carry[i] : px;
      carry[i] = __shfl_sync(kAll, xe[3 + 8 - kState + i], 31);
    }
    const bool valid = t0 < T;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float p = b[0];
      p = fmaf(w0, xe[u], p);
      p = fmaf(w1, xe[u + 1], p);
      p = fmaf(w2, xe[u + 2], p);
      p = fmaf(w3, xe[u + 3], p);
      gp[u] = valid ? act_bwd<ACT>(p, gv[u]) : 0.0f;
    }
    if (valid) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        aw[0] = fmaf(gp[u], xe[u], aw[0]);
        aw[1] = fmaf(gp[u], xe[u + 1], aw[1]);
        aw[2] = fmaf(gp[u], xe[u + 2], aw[2]);
        aw[3] = fmaf(gp[u], xe[u + 3], aw[3]);
        ab += gp[u];
      }
    }
  };

  const typename VT::Raw zero = make_uint4(0, 0, 0, 0);
  auto ld = [&](const uint16_t* r, int64_t t) { return t < T ? VT::ld(r + t) : zero; };
  float gp_cur[8];
  chunk_gp(lane * 8, ld(xr, lane * 8), ld(gr, lane * 8), gp_cur);
  typename VT::Raw xn = ld(xr, 256 + lane * 8), gn = ld(gr, 256 + lane * 8);
  for (int64_t base = 0; base < T; base += 256) {
    const int64_t t0 = base + lane * 8;
    const typename VT::Raw xnn = ld(xr, t0 + 512), gnn = ld(gr, t0 + 512);  // two chunks ahead
    float gp_next[8];
    chunk_gp(t0 + 256, xn, gn, gp_next);
    xn = xnn;
    gn = gnn;
    // gp2 of the three tokens after this lane's chunk
    float ga[kState];
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      const float down = __shfl_down_sync(kAll, gp_cur[i], 1);
      const float wrap = __shfl_sync(kAll, gp_next[i], 0);
      ga[i] = lane == 31 ? wrap : down;
    }
    if (t0 < T) {
      const float g11[11] = {gp_cur[0], gp_cur[1], gp_cur[2], gp_cur[3], gp_cur[4], gp_cur[5],
                             gp_cur[6], gp_cur[7], ga[0], ga[1], ga[2]};
      // dx[t0 + u] = w3 gp[u] + w2 gp[u+1] + w1 gp[u+2] + w0 gp[u+3] (halved weights)
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float acc = w3 * g11[u];
        acc = fmaf(w2, g11[u + 1], acc);
        acc = fmaf(w1, g11[u + 2], acc);
        acc = fmaf(w0, g11[u + 3], acc);
        v[u] = acc;
      }
      if (a.dfin && t0 + 8 == T) {  // the last three positions take dfinal_states
#pragma unroll
        for (int i = 0; i < kState; ++i) {
          const int64_t k = state_slot(row, i, a.sw);
          if (k >= 0) v[8 - kState + i] += bf16_to_f32(__ldg(a.dfin + k));
        }
      }
      VT::st(dxr + t0, VT::pack(v));
      if (t0 == 0 && a.dinit) {  // dinit[j + 3] = dxe[j], j = -3 .. -1 (gp before 0 is zero)
        const float g3[kState + 3] = {0.0f, 0.0f, 0.0f, gp_cur[0], gp_cur[1], gp_cur[2]};
#pragma unroll
        for (int i = 0; i < kState; ++i) {
          float acc = w3 * g3[i];
          acc = fmaf(w2, g3[i + 1], acc);
          acc = fmaf(w1, g3[i + 2], acc);
          acc = fmaf(w0, g3[i + 3], acc);
          const int64_t k = state_slot(row, i, a.sw);
          if (k >= 0) a.dinit[k] = f32_to_bf16(acc);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) gp_cur[u] = gp_next[u];
  }
  pdl_release();
  // the sums are of gp2 = 2 gp: halve them (exact)
  float vs[kWidth + 1] = {0.5f * aw[0], 0.5f * aw[1], 0.5f * aw[2], 0.5f * aw[3], 0.5f * ab};
#pragma unroll
  for (int k = 0; k < kWidth + 1; ++k)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) vs[k] += __shfl_xor_sync(kAll, vs[k], off);
  if (lane == 0) {
    for (int k = 0; k < kWidth + 1; ++k) a.ws[(int64_t(bb) * a.D + d) * (kWidth + 1) + k] = vs[k];
  }
}

// bwd_bdt8_kernel's pipelined walk over two adjacent channel rows (d, d + 1)
// of one batch at once (D even): each lane loads 8 tokens of x and grad_out
// of both rows per step and computes the two channels as the two halves of
// paired FP32 instructions, so one instruction serves two channels and the
// per-step addresses, halo shuffles and loop are shared.  Per channel the
// operations and their order are bwd_bdt8_kernel's, and so are the results.
// Capped at 124 registers (four 128-thread blocks per SM).  Measured: faster
// on long rows (8 x 5120 x 8192: 386 -> 368 us), slower on short ones (4 x
// 1536 x 2048: 23.8 -> 24.2 us), so the call takes it for rows of at least
// kBdtPairMinTokens tokens.
template <int ACT>
__global__ void __launch_bounds__(kBdtPairThreads, 4) bwd_bdt8x2_kernel(BwdArgs a) {
  pdl_wait();  // inputs may come from the previous kernel in the stream
  using VT = Vec<8>;
  using Raw = typename VT::Raw;
  const unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t pr = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (pr >= int64_t(a.B) * (a.D / 2)) return;  // the whole warp shares the row pair
  const int64_t row = 2 * pr;                   // rows row, row + 1 of one batch
  const int bb = int(row / a.D), d = int(row % a.D);
  float2 w[kWidth], b;
  {
    float wa[1][kWidth], ba[1], wb[1][kWidth], bq[1];
    load_weights_1(a.wr, d, wa, ba);
    load_weights_1(a.wr, d + 1, wb, bq);
#pragma unroll
    for (int k = 0; k < kWidth; ++k) w[k] = make_float2(wa[0][k], wb[0][k]);
    b = make_float2(ba[0], bq[0]);
  }
  const int64_t T = a.seqs.T;
  const uint16_t* xa = a.x + bb * a.x_sb + d * a.x_sd;
  const uint16_t* xb = xa + a.x_sd;
  const uint16_t* ga = a.g + bb * a.g_sb + d * a.g_sd;
  const uint16_t* gb = ga + a.g_sd;
  uint16_t* da = a.dx + bb * a.dx_sb + d * a.dx_sd;
  uint16_t* db = da + a.dx_sd;
  float2 carry[kState];  // for lane 0: xe of the three tokens before its next chunk
  {
    float ia[kState][1] = {{0.0f}, {0.0f}, {0.0f}}, ib[kState][1] = {{0.0f}, {0.0f}, {0.0f}};
    if (a.init) {
      load_state<1>(a.init, row, a.sw, ia);
      load_state<1>(a.init, row + 1, a.sw, ib);
    }
#pragma unroll
    for (int i = 0; i < kState; ++i) carry[i] = make_float2(ia[i][0], ib[i][0]);
  }
  float2 aw[kWidth] = {splat2(0.0f), splat2(0.0f), splat2(0.0f), splat2(0.0f)};
  float2 ab = splat2(0.0f);
  // gp2 of the chunk at t0 (zero for t0 >= T); accumulates the weight sums
  auto chunk_gp = [&](int64_t t0, Raw xra, Raw xrb, Raw gra, Raw grb, float2 (&gp)[8]) {
    float2 xe[11], gv[8];
    {
      float fa[8], fb[8], ha[8], hb[8];
      VT::unpack(xra, fa);
      VT::unpack(xrb, fb);
      VT::unpack(gra, ha);
      VT::unpack(grb, hb);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        xe[3 + u] = make_float2(fa[u], fb[u]);
        gv[u] = make_float2(ha[u], hb[u]);
      }
    }
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      const float2 last = xe[3 + 8 - kState + i];
      const float2 px = make_float2(__shfl_up_sync(kAll, last.x, 1), __shfl_up_sync(kAll, last.y, 1));
      xe[i] = lane == 0 ? carry[i] : px;
      carry[i] = make_float2(__shfl_sync(kAll, last.x, 31), __shfl_sync(kAll, last.y, 31));
    }
    const bool valid = t0 < T;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float2 p = b;
      p = ffma2(w[0], xe[u], p);
      p = ffma2(w[1], xe[u + 1], p);
      p = ffma2(w[2], xe[u + 2], p);
      p = ffma2(w[3], xe[u + 3], p);
      gp[u] = valid ? act_bwd2<ACT>(p, gv[u]) : splat2(0.0f);
    }
    if (valid) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        aw[0] = ffma2(gp[u], xe[u], aw[0]);
        aw[1] = ffma2(gp[u], xe[u + 1], aw[1]);
        aw[2] = ffma2(gp[u], xe[u + 2], aw[2]);
        aw[3] = ffma2(gp[u], xe[u + 3], aw[3]);
        ab = fadd2(ab, gp[u]);
      }
    }
  };
  const Raw zero = make_uint4(0, 0, 0, 0);
  auto ld = [&](const uint16_t* r, int64_t t) { return t < T ? VT::ld(r + t) : zero; };
  float2 gp_cur[8];
  chunk_gp(lane * 8, ld(xa, lane * 8), ld(xb, lane * 8), ld(ga, lane * 8), ld(gb, lane * 8), gp_cur);
  Raw nxa = ld(xa, 256 + lane * 8), nxb = ld(xb, 256 + lane * 8);
  Raw nga = ld(ga, 256 + lane * 8), ngb = ld(gb, 256 + lane * 8);
  for (int64_t base = 0; base < T; base += 256) {
    const int64_t t0 = base + lane * 8;
    const Raw mxa = ld(xa, t0 + 512), mxb = ld(xb, t0 + 512);  // two chunks ahead
    const Raw mga = ld(ga, t0 + 512), mgb = ld(gb, t0 + 512);
    float2 gp_next[8];
    chunk_gp(t0 + 256, nxa, nxb, nga, ngb, gp_next);
    nxa = mxa;
    nxb = mxb;
    nga = mga;
    ngb = mgb;
    // gp2 of the three tokens after this lane's chunk
    float2 gaft[kState];
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      const float2 down = make_float2(__shfl_down_sync(kAll, gp_cur[i].x, 1),
                                      __shfl_down_sync(kAll, gp_cur[i].y, 1));
      const float2 wrap = make_float2(__shfl_sync(kAll, gp_next[i].x, 0),
                                      __shfl_sync(kAll, gp_next[i].y, 0));
      gaft[i] = lane == 31 ? wrap : down;
    }
    if (t0 < T) {
      const float2 g11[11] = {gp_cur[0], gp_cur[1], gp_cur[2], gp_cur[3], gp_cur[4], gp_cur[5],
                              gp_cur[6], gp_cur[7], gaft[0], gaft[1], gaft[2]};
      // dx[t0 + u] = w3 gp[u] + w2 gp[u+1] + w1 gp[u+2] + w0 gp[u+3] (halved weights)
      float va[8], vb[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float2 acc = fmul2(w[3], g11[u]);
        acc = ffma2(w[2], g11[u + 1], acc);
        acc = ffma2(w[1], g11[u + 2], acc);
        acc = ffma2(w[0], g11[u + 3], acc);
        va[u] = acc.x;
        vb[u] = acc.y;
      }
      if (a.dfin && t0 + 8 == T) {  // the last three positions take dfinal_states
#pragma unroll
        for (int i = 0; i < kState; ++i) {
          const int64_t ka = state_slot(row, i, a.sw), kb = state_slot(row + 1, i, a.sw);
          if (ka >= 0) va[8 - kState + i] += bf16_to_f32(__ldg(a.dfin + ka));
          if (kb >= 0) vb[8 - kState + i] += bf16_to_f32(__ldg(a.dfin + kb));
        }
      }
      VT::st(da + t0, VT::pack(va));
      VT::st(db + t0, VT::pack(vb));
      if (t0 == 0 && a.dinit) {  // dinit[j + 3] = dxe[j], j = -3 .. -1 (gp before 0 is zero)
        const float2 g3[kState + 3] = {splat2(0.0f), splat2(0.0f), splat2(0.0f),
                                       gp_cur[0], gp_cur[1], gp_cur[2]};
#pragma unroll
        for (int i = 0; i < kState; ++i) {
          float2 acc = fmul2(w[3], g3[i]);
          acc = ffma2(w[2], g3[i + 1], acc);
          acc = ffma2(w[1], g3[i + 2], acc);
          acc = ffma2(w[0], g3[i + 3], acc);
          const int64_t ka = state_slot(row, i, a.sw), kb = state_slot(row + 1, i, a.sw);
          if (ka >= 0) a.dinit[ka] = f32_to_bf16(acc.x);
          if (kb >= 0) a.dinit[kb] = f32_to_bf16(acc.y);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) gp_cur[u] = gp_next[u];
  }
  pdl_release();
  // the sums are of gp2 = 2 gp: halve them (exact); one butterfly per channel
  float vs[2][kWidth + 1] = {{0.5f * aw[0].x, 0.5f * aw[1].x, 0.5f * aw[2].x, 0.5f * aw[3].x, 0.5f * ab.x},
                             {0.5f * aw[0].y, 0.5f * aw[1].y, 0.5f * aw[2].y, 0.5f * aw[3].y, 0.5f * ab.y}};
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int k = 0; k < kWidth + 1; ++k)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) vs[c][k] += __shfl_xor_sync(kAll, vs[c][k], off);
  if (lane == 0) {
    for (int c = 0; c < 2; ++c)
      for (int k = 0; k < kWidth + 1; ++k)
        a.ws[(int64_t(bb) * a.D + d + c) * (kWidth + 1) + k] = vs[c][k];
  }
}

// dweight/dbias from R rows of FP32 partial sums ws[r][D][5].  A block takes
// 32 consecutive values in eight row classes: thread (value v, class c) adds
// rows c, c + 8, c + 16, ... in increasing order (loads issued eight at a
// time, so up to 64 rows cost one round trip), then the eight class sums of each value are added in class order --
// one fixed order for a given R, so the result is bitwise repeatable.
constexpr int kFinClasses = 8;
__global__ void __launch_bounds__(32 * kFinClasses) wgrad_finalize_kernel(const float* ws, int64_t R,
                                                                          int D, WgradOut o) {
  // The next kernel may launch once every block has loaded its partial sums
  // (not earlier: a following backward launched at this kernel's start
  // measured slower).  Chains of backward calls at 4 x 2048 x 1536: 21.25 ->
  // 21.2 us, with a width-three weight 21.4 -> 21.05 us, 16 packed sequences
  // 79.2 -> 78.9 us, time-contiguous 24.3 -> 24.0 us.
  pdl_wait();  // the backward kernel's sums
  __shared__ float part[kFinClasses][32];
  const int tx = threadIdx.x & 31, c = threadIdx.x >> 5;
  const int64_t n_val = int64_t(D) * (kWidth + 1);
  const int64_t i = int64_t(blockIdx.x) * 32 + tx;
  float s = 0.0f;
  if (i < n_val) {
    constexpr int64_t kStep = kFinClasses * 8;
    for (int64_t r0 = c; r0 < R; r0 += kStep) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t r = r0 + j * kFinClasses;
        v[j] = r < R ? __ldcg(ws + r * n_val + i) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (r0 + j * kFinClasses < R) s += v[j];
    }
  }
  pdl_release();
  part[c][tx] = s;
  __syncthreads();
  if (c != 0 || i >= n_val) return;
  float t = part[0][tx];
#pragma unroll
  for (int j = 1; j < kFinClasses; ++j) t += part[j][tx];
  const int d = int(i / (kWidth + 1)), k = int(i % (kWidth + 1));
  if (k < kWidth) {
    const int kt = k - (kWidth - o.W);  // the weight's own tap; zero taps have none
    if (kt < 0) return;
    const int64_t off = d * o.dw_sd + kt * o.dw_sk;
    if (o.dw_f32) static_cast<float*>(o.dw)[off] = t;
    else static_cast<uint16_t*>(o.dw)[off] = f32_to_bf16(t);
  } else if (o.db) {
    o.db[d * o.db_sd] = f32_to_bf16(t);
  }
}

// T == 0: dinit = dfinal (the final state is the initial state), or zero.
__global__ void bwd_empty_kernel(const uint16_t* dfin, uint16_t* dinit, int64_t n) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dinit[i] = dfin ? dfin[i] : uint16_t(0);
}

// ---- host launchers ------------------------------------------------------------

int bwd_block_threads(int vec) { return vec == 8 ? bwd_threads<8>() : vec == 4 ? bwd_threads<4>() : 256; }
int bwd_ids_block_threads(int vec) { return vec == 4 ? bwd_threads<4, true>() : kGeneralThreads; }

// Dynamic shared memory of one channel-last backward block of `threads` threads.
static size_t bwd_smem_bytes(int vec, int threads) {
  if (vec == 8) return bwd_red_bytes<8>(threads) + bwd_ring_bytes<8>(threads);
  if (vec == 4) return bwd_red_bytes<4>(threads) + bwd_ring_bytes<4>(threads);
  return bwd_red_bytes<1>(threads);
}

// Opt the vector kernels in to more than 48 KB of dynamic shared memory (once
// per context: the attribute belongs to the module loaded in a context).
static ContextCache g_bwd_attr_done;
static cudaError_t bwd_smem_attributes() {
  long long done = 0;
  if (g_bwd_attr_done.get(&done) && done) return cudaSuccess;
  cudaError_t err = cudaSuccess;
  const int b8 = int(bwd_smem_bytes(8, bwd_threads<8>())), b4 = int(bwd_smem_bytes(4, bwd_threads<4>())),
            b4i = int(bwd_smem_bytes(4, bwd_threads<4, true>()));
  for (auto f : {bwd_clv_kernel<8, kActSilu>, bwd_clv_kernel<8, kActNone>})
    if (err == cudaSuccess) err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, b8);
  for (auto f : {bwd_clv_kernel<4, kActSilu>, bwd_clv_kernel<4, kActNone>})
    if (err == cudaSuccess) err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, b4);
  for (auto f : {bwd_clv_kernel<4, kActSilu, true>, bwd_clv_kernel<4, kActNone, true>})
    if (err == cudaSuccess) err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, b4i);
  if (err == cudaSuccess) g_bwd_attr_done.put(1);
  return err;
}

static ContextCache g_bwd_occupancy[3];
int bwd_blocks_per_sm(int vec) {
  ContextCache& cache = g_bwd_occupancy[vec == 8 ? 0 : vec == 4 ? 1 : 2];
  long long v = 0;
  if (cache.get(&v) && v > 0) return int(v);
  int n = 0;
  const int threads = bwd_block_threads(vec);
  const size_t smem = bwd_smem_bytes(vec, threads);
  bwd_smem_attributes();
  const cudaError_t err =
      vec == 8   ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_clv_kernel<8, kActSilu>, threads, smem)
      : vec == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_clv_kernel<4, kActSilu>, threads, smem)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_cl_kernel<1, kActSilu>, threads, smem);
  if (err == cudaSuccess && n > 0) {
    cache.put(n);
    return n;
  }
  return 1;
}

static ContextCache g_bwd_ids_occupancy[2];
int bwd_ids_blocks_per_sm(int vec) {
  ContextCache& cache = g_bwd_ids_occupancy[vec == 4 ? 0 : 1];
  long long v = 0;
  if (cache.get(&v) && v > 0) return int(v);
  int n = 0;
  bwd_smem_attributes();
  const cudaError_t err =
      vec == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bwd_clv_kernel<4, kActSilu, true>,
                                                               bwd_threads<4, true>(),
                                                               bwd_smem_bytes(4, bwd_threads<4, true>()))
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     &n, bwd_cl_kernel<1, kActSilu, true>, kGeneralThreads, bwd_red_bytes<1>(kGeneralThreads));
  if (err == cudaSuccess && n > 0) {
    cache.put(n);
    return n;
  }
  return 1;
}

// Calls with per-token sequence ids: the ring kernel (4 channels a thread) or
// the general kernels, with id masks.
template <int ACT>
static cudaError_t launch_bwd_ids(const BwdArgs& a, const BwdPlan& p, bool pdl, cudaStream_t stream) {
  if (p.kind == kLayoutChannelLast) {
    dim3 block(p.tx, p.ty), grid(p.gx, p.gy);
    if (p.vec == 4) {
      const cudaError_t err = bwd_smem_attributes();
      if (err != cudaSuccess) return err;
      return launch_kernel(bwd_clv_kernel<4, ACT, true>, grid, block, bwd_smem_bytes(4, p.tx * p.ty),
                           stream, pdl, a);
    }
    return launch_kernel(bwd_cl_kernel<1, ACT, true>, grid, block, bwd_red_bytes<1>(p.tx * p.ty),
                         stream, pdl, a);
  }
  return launch_kernel(bwd_bdt_kernel<ACT, true>, dim3(p.gx), dim3(256), 0, stream, pdl, a);
}

template <int ACT>
static cudaError_t launch_bwd_act(const BwdArgs& a, const BwdPlan& p, bool pdl,
                                  cudaStream_t stream) {
  if (p.ids) return launch_bwd_ids<ACT>(a, p, pdl, stream);
  if (p.kind == kLayoutChannelLast) {
    dim3 block(p.tx, p.ty), grid(p.gx, p.gy);
    const size_t smem = bwd_smem_bytes(p.vec, p.tx * p.ty);
    if (p.vec >= 4) {
      const cudaError_t err = bwd_smem_attributes();
      if (err != cudaSuccess) return err;
    }
    if (p.vec == 8) return launch_kernel(bwd_clv_kernel<8, ACT>, grid, block, smem, stream, pdl, a);
    if (p.vec == 4) return launch_kernel(bwd_clv_kernel<4, ACT>, grid, block, smem, stream, pdl, a);
    return launch_kernel(bwd_cl_kernel<1, ACT>, grid, block, smem, stream, pdl, a);
  }
  if (p.vec == 16)
    return launch_kernel(bwd_bdt8x2_kernel<ACT>, dim3(p.gx), dim3(kBdtPairThreads), 0, stream, pdl, a);
  if (p.vec == 8) return launch_kernel(bwd_bdt8_kernel<ACT>, dim3(p.gx), dim3(256), 0, stream, pdl, a);
  return launch_kernel(bwd_bdt_kernel<ACT>, dim3(p.gx), dim3(256), 0, stream, pdl, a);
}

// The backward kernel (launched as the programmatic dependent of whatever came
// before it: it waits before reading its inputs) writes one row of partial
// weight/bias sums per block row; the finalize kernel, its own dependent, adds
// the rows in a fixed order.  With no tokens, the rows are one zero row.
cudaError_t launch_bwd(const BwdArgs& a, const BwdPlan& p, int act, const WgradOut& o,
                       int64_t partial_rows, cudaStream_t stream) {
  const int64_t n_acc = int64_t(a.D) * (kWidth + 1);
  const bool empty = a.seqs.Q == 0;
  cudaError_t err = cudaSuccess;
  if (empty) {
    err = cudaMemsetAsync(a.ws, 0, size_t(n_acc) * sizeof(float), stream);
    if (err != cudaSuccess) return err;
    const int64_t n = int64_t(a.seqs.n_seq) * a.D * a.sw;
    if (a.dinit && n > 0)
      bwd_empty_kernel<<<unsigned((n + 255) / 256), 256, 0, stream>>>(a.dfin, a.dinit, n);
  } else {
    err = act == kActSilu ? launch_bwd_act<kActSilu>(a, p, true, stream)
                          : launch_bwd_act<kActNone>(a, p, true, stream);
    if (err != cudaSuccess) return err;
  }
  const int64_t R = empty ? 1 : partial_rows;
  err = launch_kernel(wgrad_finalize_kernel, dim3(unsigned((n_acc + 31) / 32)), dim3(32 * kFinClasses),
                      0, stream, true, static_cast<const float*>(a.ws), R, a.D, o);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace ccc
