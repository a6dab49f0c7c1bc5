// Shared device helpers for the depthwise causal conv1d kernels (sm_103a).
//
// The operation (cuDNN frontend docs, "Causal Conv1d" page): per channel d,
//   out[t] = act(bias[d] + sum_{k<4} w[d,k] * xe[t-3+k])
// on the extended sequence xe (three initial-state entries, then x).  Tap 3
// multiplies the current token (POPCORNBENCH conv1d page, causal-padding
// derivation).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ccc {

constexpr int kWidth = 4;
constexpr int kState = 3;  // W - 1

constexpr int kStatusBadCuSeqlens = 7;  // == CCC_ERR_BAD_CU_SEQLENS

// ---- programmatic dependent launch -------------------------------------------
//
// Kernels launched with programmatic stream serialization (launch_kernel with
// pdl = true) may start while the previous kernel in the stream is finishing.
// pdl_wait() blocks until that kernel has completed and its writes are
// visible, so it must precede any read of memory another kernel may have
// written; pdl_release() lets the next such kernel start launching.  Both are
// no-ops for a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- BF16 <-> FP32 ---------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// ---- activation ------------------------------------------------------------

enum Act { kActNone = 0, kActSilu = 1 };

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The kernels hold the weights and the bias times one half (an exact
// scaling), so every pre-activation they form is h = p / 2, exactly the half
// of the p the full weights would give.  With t = tanh(h) from the hardware
// tanh (one MUFU operation, relative error about 2^-11):
//   silu(p)      = p * sigmoid(p) = p (1 + t) / 2 = h + h t
//   2 * silu'(p) = 2 sigmoid(p) (1 + p (1 - sigmoid(p))) = 1 + t + h (1 - t^2)
// The backward carries gp2 = 2 * grad_out * act'(p): its weight and bias sums
// are halved once at the end, and dx = sum_k w_k gp = sum_k (w_k / 2) gp2 uses
// the halved weights as they are.
template <int ACT>
__device__ __forceinline__ float act_fwd(float h) {
  if constexpr (ACT == kActSilu) {
    return fmaf(h, tanh_approx(h), h);
  } else {
    return h + h;
  }
}

// gp2 = 2 * g * act'(p) from h = p / 2 and the incoming gradient g.
template <int ACT>
__device__ __forceinline__ float act_bwd(float h, float g) {
  if constexpr (ACT == kActSilu) {
    const float t = tanh_approx(h);
    const float v = fmaf(-t, t, 1.0f);  // 1 - t^2
    const float r = fmaf(h, v, t);      // t + h (1 - t^2)
    return fmaf(g, r, g);
  } else {
    return g + g;
  }
}

// ---- channel pairs ---------------------------------------------------------------
//
// The vector kernels compute on pairs of adjacent channels held in a float2,
// with the paired FP32 instructions of sm_100+ (one instruction, two
// independent IEEE operations, each rounded exactly like its scalar form).

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// The same operations as two scalar instructions (bitwise the same results).
// A paired instruction holds the FMA pipe twice as long as a scalar one, so
// pairing only saves issue slots; the forward's short dependent chains
// measured faster split, the backward paired.
__device__ __forceinline__ float2 ffma2_split(float2 a, float2 b, float2 c) {
  return make_float2(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y));
}

// BF16 pair (one 32-bit word, low half first) <-> float2.
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) { return make_float2(bf16_lo(u), bf16_hi(u)); }
__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Pair forms: the same operations, in the same order, as act_fwd / act_bwd.
template <int ACT, bool SPLIT = false>
__device__ __forceinline__ float2 act_fwd2(float2 h) {
  if constexpr (ACT == kActSilu) {
    const float2 t = make_float2(tanh_approx(h.x), tanh_approx(h.y));
    return SPLIT ? ffma2_split(h, t, h) : ffma2(h, t, h);
  } else {
    return make_float2(h.x + h.x, h.y + h.y);
  }
}

template <int ACT>
__device__ __forceinline__ float2 act_bwd2(float2 h, float2 g) {
  if constexpr (ACT == kActSilu) {
    const float2 t = make_float2(tanh_approx(h.x), tanh_approx(h.y));
    const float2 v = ffma2(make_float2(-t.x, -t.y), t, splat2(1.0f));
    const float2 r = ffma2(h, v, t);
    return ffma2(g, r, g);
  } else {
    return fadd2(g, g);
  }
}

// ---- vectors of V consecutive channels ---------------------------------------

template <int V>
struct Vec;

template <>
struct Vec<8> {
  using Raw = uint4;  // 8 x BF16 = 16 bytes
  __device__ __forceinline__ static Raw ld(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ static void st(uint16_t* p, Raw r) {
    __stcs(reinterpret_cast<uint4*>(p), r);
  }
  __device__ __forceinline__ static void unpack(Raw r, float (&f)[8]) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
    f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z);
    f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
  }
  __device__ __forceinline__ static Raw pack(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
  __device__ __forceinline__ static void unpack2(Raw r, float2 (&f)[4]) {
    f[0] = unpack_bf16x2(r.x); f[1] = unpack_bf16x2(r.y);
    f[2] = unpack_bf16x2(r.z); f[3] = unpack_bf16x2(r.w);
  }
  __device__ __forceinline__ static Raw pack2(const float2 (&f)[4]) {
    return make_uint4(pack_bf16x2(f[0]), pack_bf16x2(f[1]), pack_bf16x2(f[2]), pack_bf16x2(f[3]));
  }
};

template <>
struct Vec<4> {
  using Raw = uint2;  // 4 x BF16 = 8 bytes
  __device__ __forceinline__ static Raw ld(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint2*>(p));
  }
  __device__ __forceinline__ static void st(uint16_t* p, Raw r) {
    __stcs(reinterpret_cast<uint2*>(p), r);
  }
  __device__ __forceinline__ static void unpack(Raw r, float (&f)[4]) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
    f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
  }
  __device__ __forceinline__ static Raw pack(const float (&f)[4]) {
    return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
  }
  __device__ __forceinline__ static void unpack2(Raw r, float2 (&f)[2]) {
    f[0] = unpack_bf16x2(r.x); f[1] = unpack_bf16x2(r.y);
  }
  __device__ __forceinline__ static Raw pack2(const float2 (&f)[2]) {
    return make_uint2(pack_bf16x2(f[0]), pack_bf16x2(f[1]));
  }
};

template <>
struct Vec<1> {
  using Raw = uint16_t;
  __device__ __forceinline__ static Raw ld(const uint16_t* p) { return __ldg(p); }
  __device__ __forceinline__ static void st(uint16_t* p, Raw r) { __stcs(p, r); }
  __device__ __forceinline__ static void unpack(Raw r, float (&f)[1]) { f[0] = bf16_to_f32(r); }
  __device__ __forceinline__ static Raw pack(const float (&f)[1]) { return f32_to_bf16(f[0]); }
};

// States are [S, D, sw] BF16 tensors, sw = W - 1 in 1..3 entries per channel
// (entry j of channel row r -- r = sequence * D + channel -- at r * sw + j).
// The kernels embed a width-W filter in width four (leading zero taps) and
// keep a three-entry window win[i] = xe[i - 3]; for sw < 3 its first 3 - sw
// entries only ever meet zero taps: they read as 0 and are never written.
// Element index of window slot i (0..2) of channel row r, or -1 when the
// state has no such entry.
__device__ __forceinline__ int64_t state_slot(int64_t r, int i, int sw) {
  const int j = i - (kState - sw);
  return j >= 0 ? r * sw + j : -1;
}

// Narrower states (W < 4), kept out of line so that the width-four kernels'
// register allocation does not carry them.
template <int V>
__device__ __noinline__ void load_state_narrow(const uint16_t* base, int64_t r, int sw,
                                               float (&win)[kState][V]) {
#pragma unroll
  for (int c = 0; c < V; ++c)
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      const int64_t k = state_slot(r + c, i, sw);
      win[i][c] = k >= 0 ? bf16_to_f32(__ldg(base + k)) : 0.0f;
    }
}

template <int V>
__device__ __noinline__ void store_state_narrow(uint16_t* base, int64_t r, int sw,
                                                const float (&win)[kState][V]) {
#pragma unroll
  for (int c = 0; c < V; ++c)
#pragma unroll
    for (int i = 0; i < kState; ++i) {
      const int64_t k = state_slot(r + c, i, sw);
      if (k >= 0) base[k] = f32_to_bf16(win[i][c]);
    }
}

// The window of V consecutive channel rows r .. r+V-1: win[i][c] = slot i of
// row r + c.  Width four (sw = 3) reads 3*V contiguous values as vectors.
template <int V>
__device__ __forceinline__ void load_state(const uint16_t* base, int64_t r, int sw,
                                           float (&win)[kState][V]) {
  if (sw != kState) {
    load_state_narrow<V>(base, r, sw, win);
    return;
  }
  const uint16_t* s = base + r * kState;
  if constexpr (V == 8) {  // 48 bytes, 16-byte aligned
    union { uint4 q[3]; uint16_t h[24]; } u;
    const uint4* p = reinterpret_cast<const uint4*>(s);
    u.q[0] = __ldg(p); u.q[1] = __ldg(p + 1); u.q[2] = __ldg(p + 2);
#pragma unroll
    for (int c = 0; c < V; ++c)
#pragma unroll
      for (int i = 0; i < kState; ++i) win[i][c] = bf16_to_f32(u.h[c * 3 + i]);
  } else if constexpr (V == 4) {  // 24 bytes, 8-byte aligned
    union { uint2 q[3]; uint16_t h[12]; } u;
    const uint2* p = reinterpret_cast<const uint2*>(s);
    u.q[0] = __ldg(p); u.q[1] = __ldg(p + 1); u.q[2] = __ldg(p + 2);
#pragma unroll
    for (int c = 0; c < V; ++c)
#pragma unroll
      for (int i = 0; i < kState; ++i) win[i][c] = bf16_to_f32(u.h[c * 3 + i]);
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c)
#pragma unroll
      for (int i = 0; i < kState; ++i) win[i][c] = bf16_to_f32(__ldg(s + c * 3 + i));
  }
}

// Writes the state entries of rows r .. r+V-1 from the window (its last sw slots).
template <int V>
__device__ __forceinline__ void store_state(uint16_t* base, int64_t r, int sw,
                                            const float (&win)[kState][V]) {
  if (sw != kState) {
    store_state_narrow<V>(base, r, sw, win);
    return;
  }
  uint16_t* s = base + r * kState;
  if constexpr (V == 8) {
    union { uint4 q[3]; uint16_t h[24]; } u;
#pragma unroll
    for (int c = 0; c < V; ++c)
#pragma unroll
      for (int i = 0; i < kState; ++i) u.h[c * 3 + i] = f32_to_bf16(win[i][c]);
    uint4* p = reinterpret_cast<uint4*>(s);
    p[0] = u.q[0]; p[1] = u.q[1]; p[2] = u.q[2];
  } else if constexpr (V == 4) {
    union { uint2 q[3]; uint16_t h[12]; } u;
#pragma unroll
    for (int c = 0; c < V; ++c)
#pragma unroll
      for (int i = 0; i < kState; ++i) u.h[c * 3 + i] = f32_to_bf16(win[i][c]);
    uint2* p = reinterpret_cast<uint2*>(s);
    p[0] = u.q[0]; p[1] = u.q[1]; p[2] = u.q[2];
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c)
#pragma unroll
      for (int i = 0; i < kState; ++i) s[c * 3 + i] = f32_to_bf16(win[i][c]);
  }
}

// Pair forms: win[i][h] = (slot i of row r + 2h, slot i of row r + 2h + 1).
template <int V>
__device__ __forceinline__ void load_state2(const uint16_t* base, int64_t r, int sw,
                                            float2 (&win)[kState][V / 2]) {
  float f[kState][V];
  load_state<V>(base, r, sw, f);
#pragma unroll
  for (int i = 0; i < kState; ++i)
#pragma unroll
    for (int h = 0; h < V / 2; ++h) win[i][h] = make_float2(f[i][2 * h], f[i][2 * h + 1]);
}

template <int V>
__device__ __forceinline__ void store_state2(uint16_t* base, int64_t r, int sw,
                                             const float2 (&win)[kState][V / 2]) {
  float f[kState][V];
#pragma unroll
  for (int i = 0; i < kState; ++i)
#pragma unroll
    for (int h = 0; h < V / 2; ++h) { f[i][2 * h] = win[i][h].x; f[i][2 * h + 1] = win[i][h].y; }
  store_state<V>(base, r, sw, f);
}

// ---- per-thread asynchronous copies, global -> shared ---------------------------
//
// cp.async moves BYTES (8 or 16) without passing through registers; a thread
// groups its copies with commit and waits until at most N of its groups are
// still in flight.  A thread that only ever reads back what it copied itself
// needs no barrier: after the wait its own copies are visible to it.
template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t smem_addr, const void* gmem) {
  static_assert(BYTES == 8 || BYTES == 16, "cp.async moves 4, 8 or 16 bytes");
  if constexpr (BYTES == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gmem) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- weights -----------------------------------------------------------------

struct WeightRef {
  const void* w;    // [D, W] BF16 or FP32, W in 2..4
  int w_f32;
  int W;            // taps; kernel tap k (0..3) is weight tap k - (4 - W), zero below 0
  int64_t w_sd, w_sk;
  const uint16_t* bias;  // [D] BF16 or nullptr
  int64_t b_sd;
  int w_vec;        // contiguous [D, 4] and bias, 16-byte aligned: read with vectors
  int w_vec3;       // contiguous [D, 3] and bias, 16-byte aligned: read with vectors
};

// Widest channel slice a block stages: 32 threads x 8 channels (the
// eight-channel backward, whose blocks may be 64 threads wide, sizes its own).
constexpr int kMaxBlockChannels = 256;

// The weight loaders below all return the weights and the bias times one half
// (see the activation section).
//
// Block-cooperative copy of the halved weights and bias of channels
// [d_base, d_base + n) into shared memory as FP32, tap-major: ws[k*n + i] is
// w[d_base + i, k] / 2 for k < 4 and ws[4*n + i] the bias / 2 (0 without one,
// or past D).  Consecutive threads read consecutive channels, so the global reads are
// coalesced for the usual [D, 4] layout.  Every thread of the block must call it.
__device__ __forceinline__ void stage_weights(const WeightRef& r, int d_base, int n, int D,
                                              float* ws) {
  const int tid = threadIdx.x + blockDim.x * (threadIdx.y + blockDim.y * threadIdx.z);
  const int nthr = blockDim.x * blockDim.y * blockDim.z;
  const int total = n * (kWidth + 1);
  // all loads of a batch are issued before any is consumed
  constexpr int kBatch = 5;
  for (int e0 = tid; e0 < total; e0 += kBatch * nthr) {
    float v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int e = e0 + j * nthr;
      v[j] = 0.0f;
      if (e < total) {
        const int k = e / n, i = e - k * n;
        const int64_t d = int64_t(d_base) + i;
        if (d < D) {
          if (k < kWidth) {
            const int kt = k - (kWidth - r.W);  // the weight's own tap
            if (kt >= 0) {
              const int64_t o = d * r.w_sd + kt * r.w_sk;
              v[j] = 0.5f * (r.w_f32 ? __ldg(static_cast<const float*>(r.w) + o)
                                     : bf16_to_f32(__ldg(static_cast<const uint16_t*>(r.w) + o)));
            }
          } else if (r.bias) {
            v[j] = 0.5f * bf16_to_f32(__ldg(r.bias + d * r.b_sd));
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (e0 + j * nthr < total) ws[e0 + j * nthr] = v[j];
  }
  __syncthreads();
}

// A thread's V channels (local index i0, a multiple of V) from the staged slice.
template <int V>
__device__ __forceinline__ void weights_from_smem(const float* ws, int n, int i0,
                                                  float (&w)[V][kWidth], float (&b)[V]) {
  if constexpr (V % 4 == 0) {
#pragma unroll
    for (int k = 0; k <= kWidth; ++k) {
#pragma unroll
      for (int c = 0; c < V; c += 4) {
        const float4 v = *reinterpret_cast<const float4*>(ws + k * n + i0 + c);
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (k < kWidth) w[c + j][k] = f[j]; else b[c + j] = f[j];
        }
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < V; ++c) {
#pragma unroll
      for (int k = 0; k < kWidth; ++k) w[c][k] = ws[k * n + i0 + c];
      b[c] = ws[kWidth * n + i0 + c];
    }
  }
}

// Pair form: w[h][k] = (w[2h, k], w[2h+1, k]), b[h] likewise.
template <int V>
__device__ __forceinline__ void weights_from_smem2(const float* ws, int n, int i0,
                                                   float2 (&w)[V / 2][kWidth], float2 (&b)[V / 2]) {
  static_assert(V % 4 == 0, "pairs are read four channels at a time");
#pragma unroll
  for (int k = 0; k <= kWidth; ++k) {
#pragma unroll
    for (int c = 0; c < V; c += 4) {
      const float4 v = *reinterpret_cast<const float4*>(ws + k * n + i0 + c);
      if (k < kWidth) {
        w[c / 2][k] = make_float2(v.x, v.y);
        w[c / 2 + 1][k] = make_float2(v.z, v.w);
      } else {
        b[c / 2] = make_float2(v.x, v.y);
        b[c / 2 + 1] = make_float2(v.z, v.w);
      }
    }
  }
}

// The contiguous bias of channels d0 .. d0+V-1 as pairs (zero without one).
template <int V>
__device__ __forceinline__ void bias_direct2(const WeightRef& r, int d0, float2 (&b)[V / 2]) {
  if (r.bias) {
    if constexpr (V == 8) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(r.bias + d0));
      b[0] = unpack_bf16x2(u.x); b[1] = unpack_bf16x2(u.y);
      b[2] = unpack_bf16x2(u.z); b[3] = unpack_bf16x2(u.w);
    } else {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(r.bias + d0));
      b[0] = unpack_bf16x2(u.x); b[1] = unpack_bf16x2(u.y);
    }
  } else {
#pragma unroll
    for (int h = 0; h < V / 2; ++h) b[h] = splat2(0.0f);
  }
}

// Weights and bias times one half (exact).
template <int V>
__device__ __forceinline__ void halve2(float2 (&w)[V / 2][kWidth], float2 (&b)[V / 2]) {
#pragma unroll
  for (int h = 0; h < V / 2; ++h) {
    b[h] = fmul2(b[h], splat2(0.5f));
#pragma unroll
    for (int k = 0; k < kWidth; ++k) w[h][k] = fmul2(w[h][k], splat2(0.5f));
  }
}

// Pair form read by each thread straight from global memory, for a contiguous
// [D, 4] weight (and contiguous bias) aligned to 16 bytes: a thread's V
// channels are 8V (BF16) or 16V (FP32) consecutive bytes, so a handful of
// 16-byte loads replace the block-wide staging (no barrier, and the loads
// overlap the first activation loads).
template <int V>
__device__ __forceinline__ void weights_direct2(const WeightRef& r, int d0,
                                                float2 (&w)[V / 2][kWidth], float2 (&b)[V / 2]) {
  static_assert(V % 4 == 0, "vector weights need four channels at a time");
  if (r.w_f32) {
    const float4* p = static_cast<const float4*>(r.w) + d0;  // one float4 per channel
    float4 c[V];
#pragma unroll
    for (int i = 0; i < V; ++i) c[i] = __ldg(p + i);
#pragma unroll
    for (int h = 0; h < V / 2; ++h) {
      w[h][0] = make_float2(c[2 * h].x, c[2 * h + 1].x);
      w[h][1] = make_float2(c[2 * h].y, c[2 * h + 1].y);
      w[h][2] = make_float2(c[2 * h].z, c[2 * h + 1].z);
      w[h][3] = make_float2(c[2 * h].w, c[2 * h + 1].w);
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(r.w) + int64_t(d0) * kWidth);
    uint4 q[V / 2];  // two channels (8 BF16) per uint4
#pragma unroll
    for (int i = 0; i < V / 2; ++i) q[i] = __ldg(p + i);
#pragma unroll
    for (int h = 0; h < V / 2; ++h) {  // q[h] = channel 2h taps 0..3, channel 2h+1 taps 0..3
      w[h][0] = make_float2(bf16_lo(q[h].x), bf16_lo(q[h].z));
      w[h][1] = make_float2(bf16_hi(q[h].x), bf16_hi(q[h].z));
      w[h][2] = make_float2(bf16_lo(q[h].y), bf16_lo(q[h].w));
      w[h][3] = make_float2(bf16_hi(q[h].y), bf16_hi(q[h].w));
    }
  }
  bias_direct2<V>(r, d0, b);
  halve2<V>(w, b);
}

// Width three, contiguous [D, 3] weight and contiguous bias, 16-byte aligned.
template <int V>
__device__ __forceinline__ void weights_direct3(const WeightRef& r, int d0,
                                                float2 (&w)[V / 2][kWidth], float2 (&b)[V / 2]) {
  static_assert(V % 4 == 0, "vector weights need four channels at a time");
  // width three: a thread's V channels are 3V consecutive taps (6V bytes of
  // BF16: 8-byte aligned for V = 4, 16 for V = 8; 12V of FP32: 16-byte
  // aligned); weight tap k is kernel tap k + 1, kernel tap 0 is zero
  float f[3 * V];
  if (r.w_f32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(r.w) + int64_t(d0) * 3);
#pragma unroll
    for (int i = 0; i < 3 * V / 4; ++i) {
      const float4 v = __ldg(p + i);
      f[4 * i] = v.x; f[4 * i + 1] = v.y; f[4 * i + 2] = v.z; f[4 * i + 3] = v.w;
    }
  } else {
    const uint2* p = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(r.w) + int64_t(d0) * 3);
#pragma unroll
    for (int i = 0; i < 3 * V / 4; ++i) {
      const uint2 v = __ldg(p + i);
      f[4 * i] = bf16_lo(v.x); f[4 * i + 1] = bf16_hi(v.x);
      f[4 * i + 2] = bf16_lo(v.y); f[4 * i + 3] = bf16_hi(v.y);
    }
  }
#pragma unroll
  for (int h = 0; h < V / 2; ++h) {
    w[h][0] = splat2(0.0f);
#pragma unroll
    for (int k = 0; k < 3; ++k) w[h][k + 1] = make_float2(f[(2 * h) * 3 + k], f[(2 * h + 1) * 3 + k]);
  }
  bias_direct2<V>(r, d0, b);
  halve2<V>(w, b);
}

// The vector loaders: width four or width three.
template <int V>
__device__ __forceinline__ void weights_direct2_any(const WeightRef& r, int d0,
                                                    float2 (&w)[V / 2][kWidth], float2 (&b)[V / 2]) {
  if (r.w_vec3) weights_direct3<V>(r, d0, w, b);
  else weights_direct2<V>(r, d0, w, b);
}

// Weights of one channel straight from global memory (warp-uniform channel:
// every lane reads the same addresses).
__device__ __forceinline__ void load_weights_1(const WeightRef& r, int64_t d, float (&w)[1][kWidth],
                                               float (&b)[1]) {
#pragma unroll
  for (int k = 0; k < kWidth; ++k) {
    const int kt = k - (kWidth - r.W);  // the weight's own tap
    const int64_t o = d * r.w_sd + kt * r.w_sk;
    w[0][k] = kt < 0 ? 0.0f
                     : 0.5f * (r.w_f32 ? __ldg(static_cast<const float*>(r.w) + o)
                                       : bf16_to_f32(__ldg(static_cast<const uint16_t*>(r.w) + o)));
  }
  b[0] = r.bias ? 0.5f * bf16_to_f32(__ldg(r.bias + d * r.b_sd)) : 0.0f;
}

// Hint: bring the 32-byte sector holding p into L2 ahead of its load.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Hint: bring `bytes` bytes from p into L2 (p 16-byte aligned, bytes a
// multiple of 16).  One instruction for a whole contiguous run.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Kernels launched as programmatic dependents may prefetch, before
// pdl_wait(), inputs whose addresses need no memory read.  A prefetch only
// moves lines into L2, the point of coherence for every SM, so the loads
// after the wait still see everything the previous kernel wrote; the gain is
// that the first loads' DRAM latency overlaps that kernel's tail.
#ifndef CCC_PREWAIT_PREFETCH
#define CCC_PREWAIT_PREFETCH 1
#endif

// ---- sequences -----------------------------------------------------------------
//
// A call's tokens form one index space q in [0, Q).  Dense calls: sequence n is
// [n*T, (n+1)*T).  Packed calls: sequence n is [cu[n], cu[n+1]) (cuDNN page:
// packed cu_seqlens, per-sequence state, no mixing across boundaries).

struct Seqs {
  const int* cu;  // packed offsets (device), nullptr when dense
  int n_seq;
  int64_t T;      // dense: tokens per sequence
  int64_t Q;      // total tokens
};

__device__ __forceinline__ int find_seq(const Seqs& s, int64_t q) {
  if (!s.cu) {
    if (q < 0x7fffffff && s.T < 0x7fffffff)  // 32-bit division when it fits
      return static_cast<int>(static_cast<uint32_t>(q) / static_cast<uint32_t>(s.T));
    return static_cast<int>(q / s.T);
  }
  int lo = 0, hi = s.n_seq;  // invariant: cu[lo] <= q < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(s.cu + mid) <= q) lo = mid; else hi = mid;
  }
  return lo;
}

// Token range [q, q_end) of thread range (segment) seg of seg_len tokens.
// With seg_per_seq > 0 (dense calls) every sequence has its own segments, the
// last one shorter, so none straddles a sequence end; otherwise segments cut
// the whole token index.
__device__ __forceinline__ void seg_range(const Seqs& s, int64_t seg, int64_t seg_len,
                                          int64_t seg_per_seq, int64_t& q, int64_t& q_end) {
  int64_t end;
  if (seg_per_seq > 0) {
    const int64_t n = seg / seg_per_seq;
    q = n * s.T + (seg - n * seg_per_seq) * seg_len;
    end = (n + 1) * s.T;
  } else {
    q = seg * seg_len;
    end = s.Q;
  }
  q_end = q + seg_len < end ? q + seg_len : end;
}

__device__ __forceinline__ void seq_bounds(const Seqs& s, int n, int64_t& lo, int64_t& hi) {
  if (!s.cu) {
    lo = int64_t(n) * s.T;
    hi = lo + s.T;
  } else {
    lo = __ldg(s.cu + n);
    hi = __ldg(s.cu + n + 1);
  }
}

// Every block checks the whole offsets array before touching memory (cuDNN page:
// first offset 0, last offset equal to the token total, strictly increasing).
// Must be reached by every thread of the block.  Returns true when malformed;
// the first thread then records the error.
__device__ __forceinline__ bool block_rejects_cu_seqlens(const Seqs& s, int* status) {
  if (!s.cu) return false;
  const int tid = threadIdx.x + blockDim.x * (threadIdx.y + blockDim.y * threadIdx.z);
  const int nthr = blockDim.x * blockDim.y * blockDim.z;
  int bad = 0;
  for (int i = tid; i < s.n_seq; i += nthr) {
    if (__ldg(s.cu + i + 1) <= __ldg(s.cu + i)) bad = 1;
  }
  if (tid == 0 && (__ldg(s.cu) != 0 || int64_t(__ldg(s.cu + s.n_seq)) != s.Q)) bad = 1;
  bad = __syncthreads_or(bad);
  if (bad && tid == 0 && status) atomicCAS(status, 0, kStatusBadCuSeqlens);
  return bad != 0;
}

// Element offsets of token q of sequence n in an activation tensor, for the
// V channels starting at the thread's channel:  off + n * seq_step + q * st.
// Dense channel-last: seq_step = batch stride - T * token stride.  Packed, or
// a time-contiguous row handled as its own stream: seq_step = 0.
struct Stream {
  int64_t off;
  int64_t seq_step;
  int64_t st;
  __device__ __forceinline__ int64_t at(int n, int64_t q) const { return off + n * seq_step + q * st; }
};

}  // namespace ccc
