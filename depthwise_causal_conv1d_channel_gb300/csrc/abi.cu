// C ABI of the depthwise causal conv1d library: argument checks, layout
// detection, aliasing checks, launch planning and dispatch.  Every check runs
// before anything is enqueued, so a rejected call writes nothing.
#include <algorithm>
#include <atomic>
#include <stdint.h>

#include "ccc_conv1d.h"
#include "launch.h"

namespace {

using ccc::kState;
using ccc::kWidth;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int next_pow2(int64_t v) {
  int p = 1;
  while (p < v && p < (1 << 30)) p <<= 1;
  return p;
}

size_t elem_size(int dtype) { return dtype == CCC_BF16 ? 2 : 4; }

bool valid_dtype(int dtype) { return dtype == CCC_BF16 || dtype == CCC_F32 || dtype == CCC_I32; }

int64_t numel(const ccc_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// Basic sanity of a descriptor: rank, non-negative sizes and strides, data
// present when the tensor is non-empty.
bool well_formed(const ccc_tensor* t, int ndim) {
  if (!t || t->ndim != ndim || !valid_dtype(t->dtype)) return false;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0 || t->stride[i] < 0) return false;
  return numel(t) == 0 || t->data != nullptr;
}

bool shape_is(const ccc_tensor* t, int64_t a, int64_t b = -1, int64_t c = -1) {
  const int64_t s[3] = {a, b, c};
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] != s[i]) return false;
  return true;
}

// [first, last) byte range the tensor's elements occupy; empty when numel == 0.
void byte_range(const ccc_tensor* t, uintptr_t& first, uintptr_t& last) {
  if (!t || numel(t) == 0) { first = last = 0; return; }
  int64_t span = 0;
  for (int i = 0; i < t->ndim; ++i) span += (t->shape[i] - 1) * t->stride[i];
  first = reinterpret_cast<uintptr_t>(t->data);
  last = first + uintptr_t((span + 1) * int64_t(elem_size(t->dtype)));
}

bool overlaps(const ccc_tensor* a, const ccc_tensor* b) {
  uintptr_t a0, a1, b0, b1;
  byte_range(a, a0, a1);
  byte_range(b, b0, b1);
  return a0 < a1 && b0 < b1 && a0 < b1 && b0 < a1;
}

// No two index tuples of the tensor share an element (needed for outputs).
bool self_disjoint(const ccc_tensor* t) {
  if (numel(t) == 0) return true;  // no elements, nothing to share
  int idx[3];
  int n = 0;
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] > 1) idx[n++] = i;
  for (int i = 1; i < n; ++i)  // insertion sort by stride (n <= 3)
    for (int j = i; j > 0 && t->stride[idx[j]] < t->stride[idx[j - 1]]; --j) {
      const int tmp = idx[j];
      idx[j] = idx[j - 1];
      idx[j - 1] = tmp;
    }
  int64_t reach = 0;  // largest offset reachable with the smaller-stride dims
  for (int j = 0; j < n; ++j) {
    const int i = idx[j];
    if (t->stride[i] <= reach) return false;
    reach += (t->shape[i] - 1) * t->stride[i];
  }
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Layout of a [B, D, T] activation.  Size-1 dims do not constrain the layout.
int layout_of(const ccc_tensor* t) {
  const bool d_unit = t->shape[1] <= 1 || t->stride[1] == 1;
  const bool t_unit = t->shape[2] <= 1 || t->stride[2] == 1;
  if (d_unit) return ccc::kLayoutChannelLast;
  if (t_unit) return ccc::kLayoutTimeContiguous;
  return -1;
}

// Effective strides with size-1 dims normalised to what the kernels expect.
void act_strides(const ccc_tensor* t, int layout, int64_t& sb, int64_t& sd, int64_t& st) {
  sb = t->shape[0] <= 1 ? 0 : t->stride[0];
  sd = t->shape[1] <= 1 ? (layout == ccc::kLayoutChannelLast ? 1 : 0) : t->stride[1];
  st = t->shape[2] <= 1 ? (layout == ccc::kLayoutTimeContiguous ? 1 : 0) : t->stride[2];
}

// State tensors: [S, D, sw] BF16 (sw = W - 1 entries per channel), contiguous.
bool state_ok(const ccc_tensor* t, int64_t S, int64_t D, int64_t sw) {
  if (!well_formed(t, 3) || t->dtype != CCC_BF16 || !shape_is(t, S, D, sw)) return false;
  if (numel(t) == 0) return true;
  return (S <= 1 || t->stride[0] == D * sw) && (D <= 1 || t->stride[1] == sw) &&
         (sw <= 1 || t->stride[2] == 1);
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// Common checks of the tensors forward and backward share.
struct Problem {
  int B = 0, D = 0;
  int64_t T = 0;
  int n_seq = 0;  // sequences (states): B, or N when packed
  bool packed = false;
  int layout = -1;
  int w_f32 = 0;
  int W = kWidth;  // filter width, 2..4 (four on the optimized route)
  int sw = kState; // state entries per channel, W - 1
  bool ids = false; // per-token sequence ids given
};

ccc_status check_common(const ccc_tensor* x, const ccc_tensor* weight, const ccc_tensor* bias,
                        const ccc_tensor* cu, const ccc_tensor* ids, const ccc_tensor* init,
                        int activation, Problem& pb) {
  if (!well_formed(x, 3) || x->dtype != CCC_BF16) return CCC_ERR_INVALID_ARG;
  if (x->shape[1] < 1) return CCC_ERR_INVALID_ARG;
  if (x->shape[0] > INT32_MAX || x->shape[1] > INT32_MAX) return CCC_ERR_UNSUPPORTED;
  pb.B = int(x->shape[0]);
  pb.D = int(x->shape[1]);
  pb.T = x->shape[2];
  pb.layout = layout_of(x);
  if (pb.layout < 0) return CCC_ERR_UNSUPPORTED;
  if (activation != CCC_ACT_NONE && activation != CCC_ACT_SILU) return CCC_ERR_INVALID_ARG;

  if (!weight || weight->ndim != 2) return CCC_ERR_INVALID_ARG;
  if (!well_formed(weight, 2) || weight->shape[0] != pb.D) return CCC_ERR_INVALID_ARG;
  if (weight->shape[1] < 2 || weight->shape[1] > kWidth) return CCC_ERR_UNSUPPORTED;  // W in 2..4
  if (weight->dtype != CCC_BF16 && weight->dtype != CCC_F32) return CCC_ERR_INVALID_ARG;
  pb.w_f32 = weight->dtype == CCC_F32;
  pb.W = int(weight->shape[1]);
  pb.sw = pb.W - 1;

  if (bias) {
    if (!well_formed(bias, 1) || bias->dtype != CCC_BF16 || !shape_is(bias, pb.D))
      return CCC_ERR_INVALID_ARG;
    if (pb.w_f32) return CCC_ERR_UNSUPPORTED;  // FP32 weight with bias declines
  }

  pb.packed = cu != nullptr;
  if (pb.packed) {
    if (!well_formed(cu, 1) || cu->dtype != CCC_I32 || cu->shape[0] < 2) return CCC_ERR_INVALID_ARG;
    if (cu->stride[0] != 1) return CCC_ERR_UNSUPPORTED;
    if (pb.B != 1 || pb.T > INT32_MAX || cu->shape[0] - 1 > INT32_MAX) return CCC_ERR_UNSUPPORTED;
    if (pb.T == 0) return CCC_ERR_INVALID_ARG;  // N >= 1 non-empty sequences need tokens
    pb.n_seq = int(cu->shape[0] - 1);
  } else {
    pb.n_seq = pb.B;
  }
  if (ids) {
    // per-token sequence ids [B, T] int32, any non-negative strides; the page
    // makes them mutually exclusive with cu_seqlens, and no state is defined
    // with them
    if (!well_formed(ids, 2) || ids->dtype != CCC_I32 || !shape_is(ids, pb.B, pb.T))
      return CCC_ERR_INVALID_ARG;
    if (pb.packed) return CCC_ERR_INVALID_ARG;
    if (init) return CCC_ERR_UNSUPPORTED;
    pb.ids = true;
  }
  if (init && !state_ok(init, pb.n_seq, pb.D, pb.sw)) return CCC_ERR_INVALID_ARG;
  return CCC_OK;
}

bool same_act_shape(const ccc_tensor* t, const Problem& pb) {
  return well_formed(t, 3) && t->dtype == CCC_BF16 && shape_is(t, pb.B, pb.D, pb.T);
}

bool aligned(const void* p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }

// Whether vectors of V channels (2V bytes) can serve every channel-last tensor:
// every row start and every state block must be 2V-byte aligned (state blocks
// of V channels are 6V bytes; 8 bytes suffices for V = 4).
bool vec_ok(int V, const Problem& pb, std::initializer_list<const ccc_tensor*> acts,
            std::initializer_list<const ccc_tensor*> states) {
  if (pb.layout != ccc::kLayoutChannelLast || pb.D % V != 0) return false;
  for (const ccc_tensor* t : acts) {
    int64_t sb, sd, st;
    act_strides(t, pb.layout, sb, sd, st);
    if (!aligned(t->data, 2 * V) || sb % V != 0 || st % V != 0) return false;
  }
  for (const ccc_tensor* t : states)
    if (t && !aligned(t->data, V == 8 ? 16 : 8)) return false;
  return true;
}

#ifndef CCC_BWD_VEC
#define CCC_BWD_VEC 0  // 0: chosen per call by bwd_preferred_vec
#endif

// Backward vector width.  Eight channels a thread halve the per-token load,
// address and prefetch work but need ~240 registers (one 256-thread block an
// SM); four channels fit two 256-thread blocks.  Long per-thread token ranges
// favour eight, short ones the extra parallelism of four.
int bwd_preferred_vec(int64_t Q, int D, int sm_count) {
  if (CCC_BWD_VEC) return CCC_BWD_VEC;
  const int64_t resident_threads =
      int64_t(sm_count) * ccc::bwd_blocks_per_sm(8) * ccc::bwd_block_threads(8);
  const int64_t tokens_per_thread = Q * ((D + 7) / 8) / std::max<int64_t>(resident_threads, 1);
  return tokens_per_thread >= 128 ? 8 : 4;
}

// Time-contiguous dense tensors whose rows are 16-byte aligned runs of a
// multiple of 8 tokens: the warp-per-row kernels take 8 tokens a lane.
bool bdt_vec_ok(const Problem& pb, std::initializer_list<const ccc_tensor*> acts) {
  if (pb.layout != ccc::kLayoutTimeContiguous || pb.packed || pb.T % 8 != 0) return false;
  for (const ccc_tensor* t : acts) {
    int64_t sb, sd, st;
    act_strides(t, pb.layout, sb, sd, st);
    if (!aligned(t->data, 16) || sb % 8 != 0 || sd % 8 != 0 || st != 1) return false;
  }
  return true;
}

// Time-contiguous backward: 16-byte token chunks over pairs of channel rows
// (vec 16) for an even D and rows of at least kBdtPairMinTokens tokens, one
// row a warp (vec 8) for other aligned rows, else the per-token kernel (1).
int bdt_bwd_vec(const Problem& pb, std::initializer_list<const ccc_tensor*> acts) {
  if (!bdt_vec_ok(pb, acts)) return 1;
  return pb.D % 2 == 0 && pb.T >= ccc::kBdtPairMinTokens ? 16 : 8;
}

// Channels per thread: the preferred width when the tensors allow it, else 4,
// else 1 (scalar).
int pick_vec(int preferred, const Problem& pb, std::initializer_list<const ccc_tensor*> acts,
             std::initializer_list<const ccc_tensor*> states) {
  if (vec_ok(preferred, pb, acts, states)) return preferred;
  if (preferred != 4 && vec_ok(4, pb, acts, states)) return 4;
  return 1;
}

ccc::WeightRef weight_ref(const ccc_tensor* weight, const ccc_tensor* bias) {
  ccc::WeightRef r{};
  r.w = weight->data;
  r.w_f32 = weight->dtype == CCC_F32;
  r.w_sd = weight->stride[0];
  r.w_sk = weight->stride[1];
  r.W = int(weight->shape[1]);
  r.bias = bias ? static_cast<const uint16_t*>(bias->data) : nullptr;
  r.b_sd = bias ? bias->stride[0] : 0;
  const int64_t D = weight->shape[0];
  const bool bias_vec = !bias || ((D <= 1 || r.b_sd == 1) && aligned16(bias->data));
  r.w_vec = r.W == kWidth && (D <= 1 || r.w_sd == kWidth) && r.w_sk == 1 && aligned16(weight->data) &&
            bias_vec;
  r.w_vec3 = r.W == 3 && (D <= 1 || r.w_sd == 3) && (r.W <= 1 || r.w_sk == 1) &&
             aligned16(weight->data) && bias_vec;
  return r;
}

// Element strides of the [B, T] ids (size-1 dims contribute nothing).
void ids_strides(const ccc_tensor* ids, int64_t& sb, int64_t& st) {
  sb = ids && ids->shape[0] > 1 ? ids->stride[0] : 0;
  st = ids && ids->shape[1] > 1 ? ids->stride[1] : 0;
}

ccc::Seqs seqs_of(const Problem& pb, const ccc_tensor* cu) {
  ccc::Seqs s{};
  s.cu = pb.packed ? static_cast<const int*>(cu->data) : nullptr;
  s.n_seq = pb.n_seq;
  s.T = pb.T;
  s.Q = pb.packed ? pb.T : int64_t(pb.B) * pb.T;
  return s;
}

}  // namespace

namespace ccc {

// Channel-last launch shape: a block is (tx channel groups) x (ty token ranges);
// the token ranges are sized so the grid holds about `waves` full waves of
// resident blocks, each range at least `min_seg` tokens long.
#ifndef CCC_SEG_PER_SEQ
#define CCC_SEG_PER_SEQ 1  // 0: dense segments over the whole token index too
#endif
static FwdPlan plan_cl(int vec, int64_t Q, int D, int sm_count, int blocks_per_sm, int waves,
                       int64_t min_seg, int threads, int64_t seg_multiple = 1, int max_tx = 32,
                       int64_t T_seq = 0) {
  FwdPlan p{};
  p.kind = kLayoutChannelLast;
  p.vec = vec;
  const int64_t G = ceil_div(D, vec);
  p.tx = int(std::min<int64_t>(max_tx, next_pow2(G)));
  p.ty = threads / p.tx;
  p.gx = unsigned(ceil_div(G, p.tx));
  const int64_t want = std::max<int64_t>(1, int64_t(sm_count) * std::max(1, blocks_per_sm) * waves);
  int64_t gy = std::max<int64_t>(1, want / p.gx);
  int64_t seg = std::max<int64_t>(min_seg, ceil_div(std::max<int64_t>(Q, 1), gy * p.ty));
  seg = ceil_div(seg, seg_multiple) * seg_multiple;
  int64_t n_seg = ceil_div(std::max<int64_t>(Q, 1), seg);
  gy = ceil_div(n_seg, p.ty);
  if (gy > 65535) {
    seg = ceil_div(ceil_div(Q, int64_t(65535) * p.ty), seg_multiple) * seg_multiple;
    n_seg = ceil_div(Q, seg);
    gy = ceil_div(n_seg, p.ty);
  }
  // Dense calls: segments per sequence, so that no thread's range straddles a
  // sequence end (such a thread restarts its ring and steps the sequence ends
  // one token at a time, and the call waits for it), when that fits the same
  // block rows the plan asked for at the same segment length.
  p.seg_per_seq = 0;
  if (CCC_SEG_PER_SEQ && T_seq > 0 && Q > T_seq && Q % T_seq == 0) {
    const int64_t sps = ceil_div(T_seq, seg);
    const int64_t n2 = (Q / T_seq) * sps;
    const int64_t gy2 = ceil_div(n2, p.ty);
    if (gy2 <= std::max<int64_t>(gy, want / p.gx) && gy2 <= 65535) {
      p.seg_per_seq = sps;
      n_seg = n2;
      gy = gy2;
    }
  }
  p.gy = unsigned(gy);
  p.seg_len = seg;
  p.n_seg = n_seg;
  return p;
}

static FwdPlan plan_bdt(int64_t rows) {
  FwdPlan p{};
  p.kind = kLayoutTimeContiguous;
  p.vec = 1;
  p.tx = 256;
  p.ty = 1;
  p.gx = unsigned(ceil_div(std::max<int64_t>(rows, 1), 8));  // 8 warps, one row each
  p.gy = 1;
  return p;
}

FwdPlan plan_fwd(int kind, int vec, int64_t Q, int D, int64_t rows, int sm_count, bool ids,
                 int64_t T_seq) {
  if (ids) {  // kernels with id masks: the ring kernel (vec 4) or the general ones
    FwdPlan p = kind == kLayoutTimeContiguous ? plan_bdt(rows)
                : vec == 4 ? plan_cl(4, Q, D, sm_count, fwd_ids_blocks_per_sm(4), 1, 12, kFwdIdsThreads,
                                     kFwdGroupLong, 32, T_seq)
                           : plan_cl(vec, Q, D, sm_count, fwd_ids_blocks_per_sm(vec), 1, 12,
                                     kGeneralThreads, 1, 32, T_seq);
    p.ids = 1;
    p.group = kFwdGroupLong;
    if (kind == kLayoutTimeContiguous) p.vec = 1;
    return p;
  }
  if (kind == kLayoutTimeContiguous) {
    FwdPlan p = plan_bdt(rows);
    p.vec = vec;  // 8: 16-byte token chunks per lane
    return p;
  }
  // segments of a multiple of six tokens: the vector kernel's ring groups then
  // cover a segment inside a sequence exactly.  Long per-thread ranges run in
  // several waves of shorter segments, one wave per 64 tokens a thread would
  // get in one wave, up to eight (measured: 4x2048x1536 best in one wave,
  // packed 16 x U[1,4096] x 2048 in two, 8x8192x5120 in eight).
  const int bps = fwd_blocks_per_sm(vec);
  const int64_t groups = ceil_div(D, vec);
  const int64_t threads = int64_t(sm_count) * std::max(1, bps) * kFwdThreads;
  const int64_t per_thread = ceil_div(std::max<int64_t>(Q, 1) * groups, std::max<int64_t>(threads, 1));
  const int waves = int(std::min<int64_t>(8, std::max<int64_t>(1, per_thread / 64)));
  const int group = per_thread < kFwdShortTokens ? kFwdGroupShort : kFwdGroupLong;
  FwdPlan p = plan_cl(vec, Q, D, sm_count, bps, waves, 12, vec == 4 ? kFwdThreads : kGeneralThreads,
                      vec == 4 ? group : 1, 32, T_seq);
  p.group = group;
  return p;
}

BwdPlan plan_bwd(int kind, int vec, int64_t Q, int D, int64_t rows, int sm_count, bool ids,
                 int64_t T_seq) {
  if (ids) {  // kernels with id masks: the ring kernel (vec 4) or the general ones
    BwdPlan p = kind == kLayoutTimeContiguous ? plan_bdt(rows)
                : vec == 4 ? plan_cl(4, Q, D, sm_count, bwd_ids_blocks_per_sm(4), 1, 18,
                                     bwd_ids_block_threads(4), 3, 32, T_seq)
                           : plan_cl(vec, Q, D, sm_count, bwd_ids_blocks_per_sm(vec), 1, 18,
                                     kGeneralThreads, 1, 32, T_seq);
    p.ids = 1;
    if (kind == kLayoutTimeContiguous) p.vec = 1;
    return p;
  }
  if (kind == kLayoutTimeContiguous) {
    if (vec == 16) {  // a warp per pair of channel rows
      BwdPlan p{};
      p.kind = kLayoutTimeContiguous;
      p.vec = 16;
      p.tx = kBdtPairThreads;
      p.ty = 1;
      p.gx = unsigned(ceil_div(std::max<int64_t>(rows / 2, 1), kBdtPairThreads / 32));
      p.gy = 1;
      return p;
    }
    BwdPlan p = plan_bdt(rows);
    p.vec = vec;  // 8: 16-byte token chunks per lane
    return p;
  }
  // segments of a multiple of three tokens: the vector kernel's steady groups
  // of three then cover a whole segment inside a sequence, head and tail included
  const BwdPlan p = plan_cl(vec, Q, D, sm_count, bwd_blocks_per_sm(vec), 1, 18, bwd_block_threads(vec), 3,
                            32, T_seq);
  if (vec == 8) {
    // Blocks two warps wide along channels (512 channels) when that puts more
    // blocks in the wave: 8 x 5120 x 8192 takes 10 x 15 blocks instead of 20 x 7
    // (302 against 308 us); where both fill the SMs, 32 lanes wide measured
    // faster (16 packed sequences at D = 2048: 78.4 against 79.8 us).
    const BwdPlan w = plan_cl(vec, Q, D, sm_count, bwd_blocks_per_sm(vec), 1, 18, bwd_block_threads(vec), 3,
                              64, T_seq);
    if (int64_t(w.gx) * w.gy > int64_t(p.gx) * p.gy) return w;
  }
  return p;
}

int64_t bwd_partial_rows(const BwdPlan& p, int B, bool packed) {
  if (p.kind == kLayoutTimeContiguous) return packed ? 1 : std::max(B, 1);
  return p.gy;
}

}  // namespace ccc

extern "C" {

int ccc_conv1d_abi_version(void) { return CCC_CONV1D_ABI_VERSION; }

const char* ccc_status_string(int status) {
  switch (status) {
    case CCC_OK: return "ok";
    case CCC_ERR_INVALID_ARG: return "invalid argument";
    case CCC_ERR_UNSUPPORTED: return "unsupported (declined) configuration";
    case CCC_ERR_ALIAS: return "an output overlaps an input or another output";
    case CCC_ERR_NONDETERMINISTIC: return "no deterministic route for a call with bias";
    case CCC_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case CCC_ERR_CUDA: return "CUDA error";
    case CCC_ERR_BAD_CU_SEQLENS: return "malformed cu_seqlens";
    case CCC_ERR_SCRATCH_LIMIT: return "problem exceeds the built-in scratch of ccc_conv1d_bwd_noalloc";
    case CCC_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
  }
}

ccc_status ccc_conv1d_fwd(const ccc_tensor* x, const ccc_tensor* weight, const ccc_tensor* bias,
                          const ccc_tensor* cu_seqlens, const ccc_tensor* seq_idx,
                          const ccc_tensor* initial_states, const ccc_tensor* out,
                          const ccc_tensor* final_states, int activation, int* d_status,
                          cudaStream_t stream) {
  Problem pb;
  ccc_status st = check_common(x, weight, bias, cu_seqlens, seq_idx, initial_states, activation, pb);
  if (st != CCC_OK) return st;
  if (!same_act_shape(out, pb)) return CCC_ERR_INVALID_ARG;
  if (layout_of(out) != pb.layout || !self_disjoint(out)) return CCC_ERR_UNSUPPORTED;
  if (final_states && !state_ok(final_states, pb.n_seq, pb.D, pb.sw)) return CCC_ERR_INVALID_ARG;
  if (final_states && pb.ids) return CCC_ERR_UNSUPPORTED;  // no state with seq_idx
  // final_states must not share memory with the inputs (cuDNN page, aliasing rule);
  // neither may out.
  for (const ccc_tensor* in : {x, weight, bias, cu_seqlens, seq_idx, initial_states}) {
    if (!in) continue;
    if ((final_states && overlaps(final_states, in)) || overlaps(out, in)) return CCC_ERR_ALIAS;
  }
  if (final_states && overlaps(final_states, out)) return CCC_ERR_ALIAS;

  const int sms = device_sm_count();
  if (sms <= 0) return CCC_ERR_CUDA;
  ccc::FwdArgs a{};
  a.x = static_cast<const uint16_t*>(x->data);
  a.out = static_cast<uint16_t*>(out->data);
  act_strides(x, pb.layout, a.x_sb, a.x_sd, a.x_st);
  act_strides(out, pb.layout, a.o_sb, a.o_sd, a.o_st);
  a.wr = weight_ref(weight, bias);
  a.init = initial_states ? static_cast<const uint16_t*>(initial_states->data) : nullptr;
  a.fin = final_states ? static_cast<uint16_t*>(final_states->data) : nullptr;
  a.sw = pb.sw;
  a.seqs = seqs_of(pb, cu_seqlens);
  a.ids = pb.ids ? static_cast<const int*>(seq_idx->data) : nullptr;
  ids_strides(pb.ids ? seq_idx : nullptr, a.ids_sb, a.ids_st);
  a.B = pb.B;
  a.D = pb.D;
  a.status = d_status;
  if (pb.n_seq == 0) return CCC_OK;
  const int vec = pb.layout == ccc::kLayoutTimeContiguous
                      ? (bdt_vec_ok(pb, {x, out}) && !pb.ids ? 8 : 1)
                      : pick_vec(4, pb, {x, out}, {initial_states, final_states});
  const int64_t rows = pb.packed ? pb.D : int64_t(pb.B) * pb.D;
  const ccc::FwdPlan p = ccc::plan_fwd(pb.layout, vec, a.seqs.Q, pb.D, rows, sms, pb.ids,
                                       pb.packed ? 0 : pb.T);
  a.seg_len = p.seg_len;
  a.n_seg = p.n_seg;
  a.seg_per_seq = p.seg_per_seq;
  return ccc::launch_fwd(a, p, activation, stream) == cudaSuccess ? CCC_OK : CCC_ERR_CUDA;
}

// Shared by the size query and the call itself, so both agree.
static bool bwd_plan_for(const Problem& pb, int vec, bool ids, ccc::BwdPlan& p) {
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  const int64_t Q = pb.packed ? pb.T : int64_t(pb.B) * pb.T;
  const int64_t rows = pb.packed ? pb.D : int64_t(pb.B) * pb.D;
  p = ccc::plan_bwd(pb.layout, vec, Q, pb.D, rows, sms, ids, pb.packed ? 0 : pb.T);
  return true;
}

static size_t bwd_ws_bytes(const ccc::BwdPlan& p, const Problem& pb, int deterministic) {
  (void)deterministic;  // both modes write per-block partial rows
  const int64_t rows = ccc::bwd_partial_rows(p, pb.B, pb.packed);
  return size_t(std::max<int64_t>(rows, 1)) * size_t(pb.D) * (kWidth + 1) * sizeof(float);
}

size_t ccc_conv1d_bwd_workspace_size(const ccc_tensor* x, int deterministic) {
  if (!well_formed(x, 3) || x->dtype != CCC_BF16 || x->shape[1] < 1) return 0;
  if (x->shape[0] > INT32_MAX || x->shape[1] > INT32_MAX) return 0;
  Problem pb;
  pb.B = int(x->shape[0]);
  pb.D = int(x->shape[1]);
  pb.T = x->shape[2];
  pb.layout = layout_of(x);
  if (pb.layout < 0) return 0;
  // The call picks its vector width from the alignment of all its tensors, and
  // a packed call needs no more than a dense one: cover every width, with and
  // without per-token sequence ids.
  size_t n = 0;
  for (int vec : {8, 4, 1}) {
    ccc::BwdPlan p{};
    if (!bwd_plan_for(pb, vec, false, p)) return 0;
    n = std::max(n, bwd_ws_bytes(p, pb, deterministic));
    if (vec == 8) continue;
    if (!bwd_plan_for(pb, vec, true, p)) return 0;
    n = std::max(n, bwd_ws_bytes(p, pb, deterministic));
  }
  return (n + 255) / 256 * 256;
}

ccc_status ccc_conv1d_bwd(const ccc_tensor* x, const ccc_tensor* weight, const ccc_tensor* bias,
                          const ccc_tensor* cu_seqlens, const ccc_tensor* seq_idx,
                          const ccc_tensor* initial_states, const ccc_tensor* dout,
                          const ccc_tensor* dfinal_states, const ccc_tensor* dx,
                          const ccc_tensor* dweight, const ccc_tensor* dbias,
                          const ccc_tensor* dinitial_states, int activation, int deterministic,
                          void* workspace, size_t workspace_bytes, int* d_status,
                          cudaStream_t stream) {
  Problem pb;
  ccc_status st = check_common(x, weight, bias, cu_seqlens, seq_idx, initial_states, activation, pb);
  if (st != CCC_OK) return st;
  if (!same_act_shape(dout, pb) || !same_act_shape(dx, pb)) return CCC_ERR_INVALID_ARG;
  if (layout_of(dout) != pb.layout || layout_of(dx) != pb.layout || !self_disjoint(dx))
    return CCC_ERR_UNSUPPORTED;
  if (dfinal_states && !state_ok(dfinal_states, pb.n_seq, pb.D, pb.sw)) return CCC_ERR_INVALID_ARG;
  if (dfinal_states && pb.ids) return CCC_ERR_UNSUPPORTED;  // no state with seq_idx
  if (!dweight || !well_formed(dweight, 2) || !shape_is(dweight, pb.D, pb.W) ||
      dweight->dtype != weight->dtype || !self_disjoint(dweight))
    return CCC_ERR_INVALID_ARG;
  if ((bias == nullptr) != (dbias == nullptr)) return CCC_ERR_INVALID_ARG;
  if (dbias && (!well_formed(dbias, 1) || dbias->dtype != CCC_BF16 || !shape_is(dbias, pb.D) ||
                !self_disjoint(dbias)))
    return CCC_ERR_INVALID_ARG;
  if (dinitial_states && (!initial_states || !state_ok(dinitial_states, pb.n_seq, pb.D, pb.sw)))
    return CCC_ERR_INVALID_ARG;
  if (deterministic != 0 && deterministic != 1) return CCC_ERR_INVALID_ARG;
  if (deterministic && bias) return CCC_ERR_NONDETERMINISTIC;

  // outputs vs inputs, and outputs vs each other
  const ccc_tensor* ins[] = {x, weight, bias, cu_seqlens, seq_idx, initial_states, dout, dfinal_states};
  const ccc_tensor* outs[] = {dx, dweight, dbias, dinitial_states};
  for (const ccc_tensor* o : outs) {
    if (!o) continue;
    for (const ccc_tensor* in : ins)
      if (in && overlaps(o, in)) return CCC_ERR_ALIAS;
  }
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (outs[i] && outs[j] && overlaps(outs[i], outs[j])) return CCC_ERR_ALIAS;

  const int sms = device_sm_count();
  if (sms <= 0) return CCC_ERR_CUDA;
  const int64_t Q = pb.packed ? pb.T : int64_t(pb.B) * pb.T;
  int vec = 1;
  if (pb.ids)  // the general kernels: four channels a thread when aligned, else one
    vec = pb.layout == ccc::kLayoutTimeContiguous ? 1 : pick_vec(4, pb, {x, dout, dx}, {});
  else if (pb.layout == ccc::kLayoutTimeContiguous)
    vec = bdt_bwd_vec(pb, {x, dout, dx});
  else
    vec = pick_vec(bwd_preferred_vec(Q, pb.D, sms), pb, {x, dout, dx},
                   {initial_states, dfinal_states, dinitial_states});
  ccc::BwdPlan p{};
  if (!bwd_plan_for(pb, vec, pb.ids, p)) return CCC_ERR_CUDA;
  const size_t need = bwd_ws_bytes(p, pb, deterministic);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return CCC_ERR_WORKSPACE;
  {
    // the workspace is an output too
    ccc_tensor wt{workspace, CCC_F32, 1, {int64_t(need / 4), 0, 0}, {1, 0, 0}};
    for (const ccc_tensor* in : ins)
      if (in && overlaps(&wt, in)) return CCC_ERR_ALIAS;
    for (const ccc_tensor* o : outs)
      if (o && overlaps(&wt, o)) return CCC_ERR_ALIAS;
  }

  ccc::BwdArgs a{};
  a.x = static_cast<const uint16_t*>(x->data);
  a.g = static_cast<const uint16_t*>(dout->data);
  a.dx = static_cast<uint16_t*>(dx->data);
  act_strides(x, pb.layout, a.x_sb, a.x_sd, a.x_st);
  act_strides(dout, pb.layout, a.g_sb, a.g_sd, a.g_st);
  act_strides(dx, pb.layout, a.dx_sb, a.dx_sd, a.dx_st);
  a.wr = weight_ref(weight, bias);
  a.init = initial_states ? static_cast<const uint16_t*>(initial_states->data) : nullptr;
  a.dfin = dfinal_states ? static_cast<const uint16_t*>(dfinal_states->data) : nullptr;
  a.dinit = dinitial_states ? static_cast<uint16_t*>(dinitial_states->data) : nullptr;
  a.sw = pb.sw;
  a.seqs = seqs_of(pb, cu_seqlens);
  a.ids = pb.ids ? static_cast<const int*>(seq_idx->data) : nullptr;
  ids_strides(pb.ids ? seq_idx : nullptr, a.ids_sb, a.ids_st);
  a.B = pb.B;
  a.D = pb.D;
  a.seg_len = p.seg_len;
  a.n_seg = p.n_seg;
  a.seg_per_seq = p.seg_per_seq;
  a.ws = static_cast<float*>(workspace);
  a.status = d_status;

  ccc::WgradOut o{};
  o.dw = dweight->data;
  o.dw_f32 = dweight->dtype == CCC_F32;
  o.W = pb.W;
  o.dw_sd = dweight->stride[0];
  o.dw_sk = dweight->stride[1];
  o.db = dbias ? static_cast<uint16_t*>(dbias->data) : nullptr;
  o.db_sd = dbias ? dbias->stride[0] : 0;
  const int64_t R = ccc::bwd_partial_rows(p, pb.B, pb.packed);
  return ccc::launch_bwd(a, p, activation, o, R, stream) == cudaSuccess ? CCC_OK : CCC_ERR_CUDA;
}

// Same data pointer, shape and strides: the call updates in place.
static bool same_view(const ccc_tensor* a, const ccc_tensor* b) {
  if (a->data != b->data || a->ndim != b->ndim || a->dtype != b->dtype) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i] || (a->shape[i] > 1 && a->stride[i] != b->stride[i])) return false;
  return true;
}

ccc_status ccc_conv1d_update(const ccc_tensor* x, const ccc_tensor* conv_state,
                             const ccc_tensor* weight, const ccc_tensor* bias,
                             const ccc_tensor* out, int activation, cudaStream_t stream) {
  if (!x || (x->ndim != 2 && x->ndim != 3)) return CCC_ERR_INVALID_ARG;
  const bool multi = x->ndim == 3;
  if (!well_formed(x, x->ndim) || x->dtype != CCC_BF16 || x->shape[1] < 1) return CCC_ERR_INVALID_ARG;
  if (x->shape[0] > INT32_MAX || x->shape[1] > INT32_MAX || (multi && x->shape[2] > INT32_MAX))
    return CCC_ERR_UNSUPPORTED;
  const int B = int(x->shape[0]), D = int(x->shape[1]);
  const int L = multi ? int(x->shape[2]) : 1;
  if (D > 1 && x->stride[1] != 1) return CCC_ERR_UNSUPPORTED;
  if (activation != CCC_ACT_NONE && activation != CCC_ACT_SILU) return CCC_ERR_INVALID_ARG;
  if (!weight || !well_formed(weight, 2) || weight->shape[0] != D) return CCC_ERR_INVALID_ARG;
  if (weight->shape[1] < 2 || weight->shape[1] > kWidth) return CCC_ERR_UNSUPPORTED;  // W in 2..4
  const int sw = int(weight->shape[1]) - 1;
  if (!state_ok(conv_state, B, D, sw)) return CCC_ERR_INVALID_ARG;
  if (weight->dtype != CCC_BF16 && weight->dtype != CCC_F32) return CCC_ERR_INVALID_ARG;
  if (bias) {
    if (!well_formed(bias, 1) || bias->dtype != CCC_BF16 || !shape_is(bias, D))
      return CCC_ERR_INVALID_ARG;
    if (weight->dtype == CCC_F32) return CCC_ERR_UNSUPPORTED;
  }
  if (!out || out->ndim != x->ndim || !well_formed(out, out->ndim) || out->dtype != CCC_BF16 ||
      !shape_is(out, B, D, multi ? L : -1))
    return CCC_ERR_INVALID_ARG;
  if ((D > 1 && out->stride[1] != 1) || !self_disjoint(out)) return CCC_ERR_UNSUPPORTED;
  for (const ccc_tensor* in : {conv_state, weight, bias})
    if (in && overlaps(out, in)) return CCC_ERR_ALIAS;
  if (overlaps(x, conv_state)) return CCC_ERR_ALIAS;
  // out either is x (in place: every element is read before its thread writes
  // it) or stays clear of it (another thread's x otherwise)
  if (overlaps(out, x) && !same_view(out, x)) return CCC_ERR_ALIAS;
  if (B == 0 || L == 0) return CCC_OK;  // nothing to compute; the state is unchanged

  ccc::UpdArgs a{};
  a.x = static_cast<const uint16_t*>(x->data);
  a.x_sb = B > 1 ? x->stride[0] : 0;
  a.x_sl = multi && L > 1 ? x->stride[2] : 0;
  a.state = static_cast<uint16_t*>(conv_state->data);
  a.sw = sw;
  a.out = static_cast<uint16_t*>(out->data);
  a.o_sb = B > 1 ? out->stride[0] : 0;
  a.o_sl = multi && L > 1 ? out->stride[2] : 0;
  a.wr = weight_ref(weight, bias);
  a.B = B;
  a.D = D;
  a.L = L;
  // vectors of V channels: 2V-byte aligned rows; a state block of V channels
  // is 6V bytes (16-byte alignment for V = 8, 8 for V = 4)
  auto fits = [&](int V) {
    return D % V == 0 && aligned(x->data, 2 * V) && aligned(out->data, 2 * V) &&
           aligned(conv_state->data, V == 8 ? 16 : 8) && a.x_sb % V == 0 && a.o_sb % V == 0 &&
           a.x_sl % V == 0 && a.o_sl % V == 0;
  };
  const int vec = fits(8) ? 8 : fits(4) ? 4 : 1;
  return ccc::launch_update(a, vec, activation, stream) == cudaSuccess ? CCC_OK : CCC_ERR_CUDA;
}

ccc_status ccc_read_status(int* d_status, cudaStream_t stream) {
  if (!d_status) return CCC_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CCC_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CCC_ERR_CUDA;
  if (h != 0 && cudaMemset(d_status, 0, sizeof(int)) != cudaSuccess) return CCC_ERR_CUDA;
  return static_cast<ccc_status>(h);
}

// ---- full-channel dilated causal conv1d -------------------------------------------

ccc_status ccc_fullconv1d_pack_weight(const ccc_tensor* weight, const ccc_tensor* packed,
                                      cudaStream_t stream) {
  if (!well_formed(weight, 3) || (weight->dtype != CCC_BF16 && weight->dtype != CCC_F32))
    return CCC_ERR_INVALID_ARG;
  const int64_t Cout = weight->shape[0], Cin = weight->shape[1], K = weight->shape[2];
  if (!well_formed(packed, 3) || packed->dtype != CCC_BF16 || !shape_is(packed, K, Cout, Cin))
    return CCC_ERR_INVALID_ARG;
  const int64_t n = K * Cout * Cin;
  if (n > 0 && !((Cin <= 1 || packed->stride[2] == 1) && (Cout <= 1 || packed->stride[1] == Cin) &&
                 (K <= 1 || packed->stride[0] == Cout * Cin)))
    return CCC_ERR_UNSUPPORTED;  // the packed weight is contiguous
  if (overlaps(weight, packed)) return CCC_ERR_ALIAS;
  if (n == 0) return CCC_OK;
  return ccc::launch_pack_weight(weight->data, weight->dtype == CCC_F32, weight->stride[0],
                                 weight->stride[1], weight->stride[2],
                                 static_cast<uint16_t*>(packed->data), Cout, Cin, K, stream) == cudaSuccess
             ? CCC_OK
             : CCC_ERR_CUDA;
}

ccc_status ccc_fullconv1d_fwd(const ccc_tensor* x, const ccc_tensor* packed_weight,
                              const ccc_tensor* bias, int dilation, const ccc_tensor* out,
                              int* d_status, cudaStream_t stream) {
  if (!well_formed(x, 3) || x->dtype != CCC_BF16) return CCC_ERR_INVALID_ARG;
  if (!well_formed(packed_weight, 3) || packed_weight->dtype != CCC_BF16) return CCC_ERR_INVALID_ARG;
  const int64_t B = x->shape[0], Cin = x->shape[1], T = x->shape[2];
  const int64_t K = packed_weight->shape[0], Cout = packed_weight->shape[1];
  if (packed_weight->shape[2] != Cin || K < 1 || Cin < 1 || Cout < 1) return CCC_ERR_INVALID_ARG;
  if (dilation < 1) return CCC_ERR_INVALID_ARG;
  if (!well_formed(out, 3) || out->dtype != CCC_BF16 || !shape_is(out, B, Cout, T))
    return CCC_ERR_INVALID_ARG;
  if (bias && (!well_formed(bias, 1) || (bias->dtype != CCC_BF16 && bias->dtype != CCC_F32) ||
               !shape_is(bias, Cout)))
    return CCC_ERR_INVALID_ARG;
  // what the tensor-memory GEMM reads: channel-last x and out with rows on
  // 16-byte boundaries, a contiguous packed weight, sizes that fit its grid
  if (Cin % 8 != 0 || Cout % 8 != 0) return CCC_ERR_UNSUPPORTED;
  if (K > 1024 || (K - 1) * int64_t(dilation) > INT32_MAX / 2 || T > INT32_MAX / 2 ||
      B > 65535 || (Cout + 255) / 256 > 65535 || Cin > (int64_t(1) << 24))
    return CCC_ERR_UNSUPPORTED;
  // the persistent kernel numbers its 256 x 256 tiles with int
  if (B * ((T + 255) / 256) * ((Cout + 255) / 256) > INT32_MAX / 2) return CCC_ERR_UNSUPPORTED;
  for (const ccc_tensor* t : {x, out}) {
    const int64_t sb = t->shape[0] > 1 ? t->stride[0] : 0;
    const int64_t st = t->shape[2] > 1 ? t->stride[2] : 0;
    if (t->shape[1] > 1 && t->stride[1] != 1) return CCC_ERR_UNSUPPORTED;
    if (sb % 8 != 0 || st % 8 != 0 || !aligned16(t->data)) return CCC_ERR_UNSUPPORTED;
    if (T > 1 && st < t->shape[1]) return CCC_ERR_UNSUPPORTED;
  }
  if (!((Cin <= 1 || packed_weight->stride[2] == 1) &&
        (Cout <= 1 || packed_weight->stride[1] == Cin) &&
        (K <= 1 || packed_weight->stride[0] == Cout * Cin)) ||
      !aligned16(packed_weight->data))
    return CCC_ERR_UNSUPPORTED;
  if (!self_disjoint(out)) return CCC_ERR_UNSUPPORTED;
  for (const ccc_tensor* in : {x, packed_weight, bias})
    if (in && overlaps(out, in)) return CCC_ERR_ALIAS;
  if (B == 0 || T == 0) return CCC_OK;

  ccc::FullConvArgs f{};
  f.x = static_cast<const uint16_t*>(x->data);
  f.x_sb = B > 1 ? x->stride[0] : 0;
  f.x_st = T > 1 ? x->stride[2] : Cin + (8 - Cin % 8) % 8;
  f.w = static_cast<const uint16_t*>(packed_weight->data);
  f.bias = bias ? bias->data : nullptr;
  f.bias_f32 = bias && bias->dtype == CCC_F32;
  f.bias_s = bias ? bias->stride[0] : 0;
  f.out = static_cast<uint16_t*>(out->data);
  f.o_sb = B > 1 ? out->stride[0] : 0;
  f.o_st = T > 1 ? out->stride[2] : 0;
  f.B = B;
  f.T = T;
  f.Cin = int(Cin);
  f.Cout = int(Cout);
  f.K = int(K);
  f.dil = dilation;
  f.status = d_status;
  return ccc::launch_fullconv(f, stream) == cudaSuccess ? CCC_OK : CCC_ERR_CUDA;
}

}  // extern "C"
