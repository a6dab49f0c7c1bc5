// Full-channel dilated causal conv1d on the 5th-generation tensor cores
// (POPCORNBENCH conv1d page: a Conv1d over all input channels with dilation,
// left-padded by P = (K-1)*dil so that tap k reads input position
// t + k*dil - P, zero before 0).  With channel-last activations and the
// weight packed tap-major as Wk[oc, ic] = W[oc, ic, k]:
//
//   out[b, t, oc] = bias[oc] + sum_k sum_ic x[b, t - (K-1-k)*dil, ic] * Wk[oc, ic]
//
// a sum of K GEMMs whose A operand is x shifted along tokens.  This is a dense
// contraction (2 * Cin * K FLOPs per output), so it runs as an implicit GEMM
// on tcgen05.  Two kernels: the persistent kernel further below serves
// receptive fields up to 256 tokens, loading one x slice per block of input
// channels for all taps; the per-tap kernel first, for longer receptive
// fields, runs one CTA per output tile of 128 tokens x 256 output channels of
// one batch row.  For each (tap, block of 64 input channels) a TMA load brings
// the 128 x 64 slice of x starting at token t0 - (K-1-k)*dil (coordinates
// before token 0 read as zeros: the causal padding needs no padded copy) and
// the 256 x 64 slice of Wk into a 4-stage ring of 128-byte-swizzled shared
// memory; one thread issues four tcgen05.mma (M 128, N 256, K 16, BF16 in,
// FP32 accumulate) into a 128 x 256 FP32 accumulator in tensor memory; after
// the last block the four warps read the accumulator back with tcgen05.ld,
// add the bias, round to BF16 and store.
//
// Every wait on an mbarrier is bounded (by the global timer): when one runs
// out, the kernel records CCC_ERR_DEVICE_TIMEOUT in the status word, waits
// (bounded again) for its own copies and MMAs in flight, frees its tensor
// memory and returns, so the context stays usable.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "ccc_conv1d.h"
#include "launch.h"

namespace ccc {
namespace fullconv {

constexpr int BM = 128;  // tokens per tile (MMA M, TMEM lanes)
constexpr int BN = 256;  // output channels per tile (MMA N, TMEM columns)
constexpr int BK = 64;   // input channels per stage: one 128-byte swizzle row of BF16
constexpr int UK = 16;   // K of one kind::f16 MMA
constexpr int kStages = 4;
constexpr int kThreads = 128;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = BN;  // FP32 accumulator: one column per output channel
// ring + barriers (2 per stage + 1) + TMEM address + abort flag + the tile's
// bias, plus slack to align the ring to 1024 bytes (the 128-byte swizzle
// repeats every 8 rows)
constexpr size_t kSmemBytes =
    1024 + size_t(kStages) * kStageBytes + 8 * (2 * kStages + 1) + 16 + size_t(BN) * 4;
constexpr int kStatusTimeout = 9;  // == CCC_ERR_DEVICE_TIMEOUT
constexpr uint64_t kWaitLimitNs = 500ull * 1000 * 1000;

// Instruction descriptor of tcgen05.mma kind::f16 for M 128 and the given N:
// D FP32 (bits 4-5 = 1), A and B BF16 (bits 7-9 = 1, 10-12 = 1), both K-major
// (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_m128(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(128 >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major tile stored as TMA writes it
// with 128-byte swizzling: rows of 64 BF16 (128 bytes), 8-row groups 1024 bytes
// apart, the 16-byte chunks of a row permuted by address bits 7-9 (the row's
// place in its 1024-byte group).  Start address >> 4 at bits 0-13; leading
// byte offset (unused for swizzled K-major tiles) 16 >> 4 at bits 16-29;
// stride byte offset 1024 >> 4 at bits 32-45; descriptor version 1 at bits
// 46-48; base offset 0 at bits 49-51; layout SWIZZLE_128B = 2 at bits 61-63.
// The tensor cores apply the permutation to the addresses they form, like the
// TMA unit does, so a matrix may start at any row of a swizzled tile (row r:
// start + 128 r) with the base offset left at 0 -- measured on sm_103a with
// an own probe over row offsets 0..16, exact for every offset.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// ---- PTX wrappers ----------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread until the phase completes or `ns`
// nanoseconds pass: a waiting thread sleeps instead of polling, so it takes no
// issue slots or shared-memory bandwidth from the producer and MMA threads.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase of `bar` with the given parity to complete; false when
// kWaitLimitNs pass first (or after 2^20 sleeps, should the timer stall).
// Inlined: as an out-of-line call it made the producer and MMA threads save
// and restore registers around every wait, which slowed the MMA stream of a
// 256 x 256 tile from 43 to 51 us.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 20); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, M 128 x N x K 16 (N from the descriptor).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct Args {
  uint16_t* out;      // [B, T, Cout] storage (channel stride 1)
  int64_t o_sb, o_st;
  const void* bias;   // [Cout] BF16 or FP32, or nullptr
  int bias_f32;
  int64_t bias_s;
  int T, Cout, K, dil;
  int n_kblk;         // blocks of 64 input channels
  int* status;
};

extern __shared__ __align__(1024) uint8_t fc_smem[];

// Bias of the tile's output channels n0 .. n0+N-1 as FP32 in shared memory
// (zero past Cout or without a bias); every thread of the block calls it.
template <int N>
__device__ __forceinline__ void stage_bias(const Args& a, int n0, float* bias_s) {
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int oc = n0 + i;
    float v = 0.0f;
    if (a.bias && oc < a.Cout)
      v = a.bias_f32 ? __ldg(static_cast<const float*>(a.bias) + int64_t(oc) * a.bias_s)
                     : bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.bias) + int64_t(oc) * a.bias_s));
    bias_s[i] = v;
  }
}

// Epilogue of one 128-row accumulator (TMEM columns col0 .. col0+N-1, rows =
// tokens t_first .. t_first+127): warp w takes TMEM lanes 32w .. 32w+31.  Each
// thread reads its row's FP32 sums 64 columns at a time (two loads in flight
// per wait), adds the bias, rounds to BF16 and writes the row piece into the
// warp's staging rows in shared memory (row stride N*2 + 16 bytes, so the
// 16-byte writes of the 32 rows spread over all banks); then the warp writes
// its 32 rows to global memory one row at a time, each row one coalesced
// N*2-byte store.  `stage` is this warp's 32 staging rows.
template <int N>
__device__ __forceinline__ void store_accumulator(const Args& a, uint32_t tmem, uint32_t col0,
                                                  int t_first, int n0, int bb, const float* bias_s,
                                                  uint8_t* stage) {
  constexpr int kRowBytes = N * 2 + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncols = a.Cout - n0 < N ? a.Cout - n0 : N;  // a multiple of 8
  for (int c0 = 0; c0 < N && c0 < ncols; c0 += 64) {  // warp-uniform bounds
    uint32_t r0[32], r1[32];
    const uint32_t taddr = tmem + (uint32_t(warp * 32) << 16) + col0 + uint32_t(c0);
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_ld_wait();
    uint8_t* row = stage + lane * kRowBytes + c0 * 2;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t* r = q < 4 ? r0 + 8 * q : r1 + 8 * (q - 4);
      const float* bq = bias_s + c0 + 8 * q;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]) + bq[j];
      *reinterpret_cast<uint4*>(row + 16 * q) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
  }
  __syncwarp();
  for (int rr = 0; rr < 32; ++rr) {
    const int t = t_first + warp * 32 + rr;
    if (t >= a.T) break;  // rows past T are the tile's tail
    uint16_t* orow = a.out + int64_t(bb) * a.o_sb + int64_t(t) * a.o_st + n0;
    const uint8_t* srow = stage + rr * kRowBytes;
    for (int cc = lane * 8; cc < ncols; cc += 256)
      *reinterpret_cast<uint4*>(orow + cc) = *reinterpret_cast<const uint4*>(srow + cc * 2);
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1)
    fullconv_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                    Args a) {
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_release();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * BM, n0 = blockIdx.y * BN, bb = blockIdx.z;
  const int n_iter = a.K * a.n_kblk;

  // shared layout: A stages, B stages (1024-aligned), then the barriers
  const uint32_t raw = smem_u32(fc_smem);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t sA = raw + pad;
  const uint32_t sB = sA + kStages * kABytes;
  const uint32_t bars = sB + kStages * kBBytes;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  const uint32_t acc_bar = bars + 8u * (2 * kStages);
  const uint32_t tmem_slot = acc_bar + 8;
  uint8_t* gbase = fc_smem + pad + (bars - sA) + 8 * (2 * kStages + 1);  // generic view of the slot
  volatile uint32_t* tmem_slot_p = reinterpret_cast<volatile uint32_t*>(gbase);
  volatile int* abort_p = reinterpret_cast<volatile int*>(gbase + 4);
  float* bias_s = reinterpret_cast<float*>(gbase + 16);  // BN floats
  stage_bias<BN>(a, n0, bias_s);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_bar, 1);
    *abort_p = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_x);
    prefetch_map(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_p;

  auto fail = [&]() {
    *abort_p = 1;
    if (a.status) atomicCAS(a.status, 0, kStatusTimeout);
  };
  // Tiles start their walk over the channel blocks at different blocks, so the
  // CTAs running at once read different weight slices instead of all asking
  // L2 for the same lines (the sum's order is fixed per tile).
  const int rot = int((blockIdx.x + blockIdx.y + blockIdx.z) % unsigned(a.n_kblk));

  if (warp == 0 && lane == 0) {
    // producer: TMA loads of the (tap, channel block) stages
    int issued = 0;
    for (int i = 0; i < n_iter; ++i) {
      const int s = i % kStages;
      const uint32_t ph = uint32_t(i / kStages) & 1u;
      if (!mbar_wait(empty_bar(s), ph ^ 1u)) {  // the MMAs have released the stage
        fail();
        break;
      }
      if (*abort_p) break;
      const int k = i / a.n_kblk, kb = (i - k * a.n_kblk + rot) % a.n_kblk;
      mbar_expect_tx(full_bar(s), kStageBytes);
      tma_load_3d(sA + s * kABytes, &map_x, full_bar(s), kb * BK, t0 - (a.K - 1 - k) * a.dil, bb);
      tma_load_3d(sB + s * kBBytes, &map_w, full_bar(s), kb * BK, n0, k);
      ++issued;
    }
    if (*abort_p) {  // let the loads in flight land before the CTA leaves
      for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
        mbar_wait(full_bar(i % kStages), uint32_t(i / kStages) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    for (int i = 0; i < n_iter; ++i) {
      const int s = i % kStages;
      const uint32_t ph = uint32_t(i / kStages) & 1u;
      if (!mbar_wait(full_bar(s), ph)) {  // both tiles of the stage have landed
        fail();
        break;
      }
      if (*abort_p) break;
      tc_fence_after();
      const uint64_t ad = sw128_desc(sA + s * kABytes), bd = sw128_desc(sB + s * kBBytes);
#pragma unroll
      for (int j = 0; j < BK / UK; ++j)  // +32 bytes along K per MMA: +2 in the address field
        mma_bf16(tmem, ad + 2 * j, bd + 2 * j, idesc_m128(BN), (i > 0 || j > 0) ? 1u : 0u);
      mma_commit(empty_bar(s));
    }
    mma_commit(acc_bar);  // all MMAs above complete (also on the abort path)
  }
  __syncwarp();

  // epilogue: the ring is idle now; warp w stages its rows at the ring's start.
  // Lane 0 waits and tells the warp, so the warp-wide tcgen05.ld is reached by
  // all lanes or by none.
  int st = 0;
  if (lane == 0) {
    st = mbar_wait(acc_bar, 0) ? (*abort_p ? 1 : 0) : 2;
    if (st == 2) fail();
  }
  st = __shfl_sync(0xffffffffu, st, 0);
  tc_fence_after();
  if (st == 0)
    store_accumulator<BN>(a, tmem, 0, t0, n0, bb, bias_s, fc_smem + pad + warp * 32 * (BN * 2 + 16));
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- persistent kernel: one x slice per channel block shared by all taps -----------
//
// The taps of one output tile read the same x rows shifted by multiples of the
// dilation, so instead of one x slice per tap, the kernel below loads per block
// of 64 input channels ONE slice of RA = 256 + pad rows (tokens t0 - pad ..
// t0 + 255, pad >= (K-1)*dil rounded up to 16) and lets tap k read it from row
// pad - (K-1-k)*dil on: the MMA's A descriptor simply starts at that row (see
// sw128_desc).  A tile is 256 tokens -- two M-128 accumulators sharing each
// weight slice -- by N output channels, so per (channel block, tap) the tensor
// cores do 2 x 128 x N x 64 multiply-adds for N x 128 bytes of weight plus a
// quarter of the x slice: about half the bytes per FLOP of the per-tap kernel.
//
// One CTA runs per SM and walks a static list of work items: whole tiles, then,
// when the tiles do not fill the last wave, the remaining tiles cut into halves
// of 128 tokens (one accumulator each), so the last wave is shorter.  (A half
// keeps all of the tile's weight bytes for half the MMAs, so it takes about
// three quarters of a tile's time, bound by L2 reads; halves of N / 2 output
// channels measured slower still, the N / 2 MMAs running below the tensor
// cores' rate.)
//
// Warp 0 issues the TMA loads, warp 1 the MMAs, warps 2-9 drain the
// accumulators: warp w reads TMEM lanes 32 (w % 4) .. +31 of accumulator
// (w - 2) / 4, adds the bias, keeps the row as packed BF16 in registers and
// releases the tensor memory before it stores, so the next item's MMAs run
// while the rows go out.  The loads of the next item fill the ring while the
// MMAs of this one finish.

struct SharedPlan {
  int ra;    // rows of an x slot (multiple of 16, at most 512)
  int pad;   // ra - 256: rows before t0
  int nb;    // weight stages
};

// Work items: [0, n_main) whole tiles (tile = item), [n_main, n_items) half
// tiles (tile n_main + j / 2, tokens 128 (j % 2) on; j = item - n_main).
// Tiles are numbered token tile fastest, then output-channel tile, then row.
struct Sched {
  int n_tb, n_ob;
  int n_main, n_items;
};

struct Item {
  int t0, n0, bb, nh;  // first token, first output channel, batch row, accumulators (M-128 halves)
};

template <int N>
__device__ __forceinline__ Item item_at(const Sched& sc, int w) {
  int tile = w, t_off = 0, nh = 2;
  if (w >= sc.n_main) {
    const int j = w - sc.n_main;
    tile = sc.n_main + (j >> 1);
    t_off = 128 * (j & 1);
    nh = 1;
  }
  const int tb = tile % sc.n_tb, r = tile / sc.n_tb;
  return Item{tb * 256 + t_off, (r % sc.n_ob) * N, r / sc.n_ob, nh};
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

constexpr int kPThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int kEpiWarps = 8;
constexpr int kChunk = 32;                            // columns per staged store round
constexpr uint32_t kStageRow = kChunk * 2 + 16;       // staging row stride: banks spread
constexpr uint32_t kStageWarp = 32 * kStageRow;       // one warp's staging rows

template <int N>
constexpr size_t persistent_fixed_smem(int ra) {
  // align slack, two x slots, epilogue staging, per-warp bias copies,
  // barriers + TMEM address + abort flag
  return 1024 + 2 * size_t(ra) * 128 + kEpiWarps * size_t(kStageWarp) + kEpiWarps * size_t(N) * 4 + 256;
}

template <int N>
__global__ void __launch_bounds__(kPThreads, 1)
    fullconv_persistent_kernel(const __grid_constant__ CUtensorMap map_x,
                               const __grid_constant__ CUtensorMap map_w, Args a, SharedPlan sp,
                               Sched sc) {
  constexpr uint32_t kBStage = uint32_t(N) * BK * 2;
  constexpr uint32_t kCols = 2 * N;  // two accumulators of N FP32 columns
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t slot_a = uint32_t(sp.ra) * 128;

  // shared layout: x slots, weight stages, staging rows, bias copies, barriers
  const uint32_t raw = smem_u32(fc_smem);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint32_t sA = raw + pad;
  const uint32_t sB = sA + 2 * slot_a;
  const uint32_t sStage = sB + uint32_t(sp.nb) * kBStage;
  const uint32_t sBias = sStage + kEpiWarps * kStageWarp;
  const uint32_t bars = sBias + kEpiWarps * N * 4;
  auto a_full = [&](int i) { return bars + 8u * i; };
  auto a_empty = [&](int i) { return bars + 8u * (2 + i); };
  auto b_full = [&](int i) { return bars + 8u * (4 + i); };
  auto b_empty = [&](int i) { return bars + 8u * (4 + sp.nb + i); };
  const uint32_t acc_full = bars + 8u * (4 + 2 * sp.nb);
  const uint32_t acc_empty = acc_full + 8;
  const uint32_t mma_done = acc_full + 16;
  const uint32_t tmem_slot = acc_full + 24;
  uint8_t* const gsm = fc_smem + pad;  // generic view of sA
  auto generic = [&](uint32_t s) { return gsm + (s - sA); };
  volatile uint32_t* tmem_slot_p = reinterpret_cast<volatile uint32_t*>(generic(tmem_slot));
  volatile int* abort_p = reinterpret_cast<volatile int*>(generic(tmem_slot) + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(a_full(i), 1);
      mbar_init(a_empty(i), 1);
    }
    for (int i = 0; i < sp.nb; ++i) {
      mbar_init(b_full(i), 1);
      mbar_init(b_empty(i), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(mma_done, 1);
    *abort_p = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_x);
    prefetch_map(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot_p;
  // The setup above reads nothing a previous kernel writes, so it runs while
  // that kernel finishes (launched as its programmatic dependent); every read
  // of x, the weight and the bias comes after this wait.
  pdl_wait();
  pdl_release();

  auto fail = [&]() {
    *abort_p = 1;
    if (a.status) atomicCAS(a.status, 0, kStatusTimeout);
  };

  if (warp == 0 && lane == 0) {
    // producer: per channel block one x slice (two boxes of ra / 2 rows),
    // then the K weight slices; runs ahead across items as far as the ring allows
    int ia = 0, ib = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < sc.n_items; w += gridDim.x) {
      const Item it = item_at<N>(sc, w);
      for (int kb = 0; ok && kb < a.n_kblk; ++kb) {
        const int sa = ia & 1;
        if (!mbar_wait(a_empty(sa), (uint32_t(ia >> 1) & 1u) ^ 1u) || *abort_p) {
          ok = false;
          break;
        }
        mbar_expect_tx(a_full(sa), slot_a);
        const uint32_t dst = sA + sa * slot_a;
        tma_load_3d(dst, &map_x, a_full(sa), kb * BK, it.t0 - sp.pad, it.bb);
        tma_load_3d(dst + slot_a / 2, &map_x, a_full(sa), kb * BK, it.t0 - sp.pad + sp.ra / 2, it.bb);
        ++ia;
        for (int k = 0; k < a.K; ++k) {
          const int s = ib % sp.nb;
          if (!mbar_wait(b_empty(s), (uint32_t(ib / sp.nb) & 1u) ^ 1u) || *abort_p) {
            ok = false;
            break;
          }
          mbar_expect_tx(b_full(s), kBStage);
          tma_load_3d(sB + s * kBStage, &map_w, b_full(s), kb * BK, it.n0, k);
          ++ib;
        }
      }
    }
    if (!ok) {  // let the loads in flight land before the CTA leaves
      if (!*abort_p) fail();
      for (int i = ia - 2 < 0 ? 0 : ia - 2; i < ia; ++i) mbar_wait(a_full(i & 1), uint32_t(i >> 1) & 1u);
      for (int i = ib - sp.nb < 0 ? 0 : ib - sp.nb; i < ib; ++i)
        mbar_wait(b_full(i % sp.nb), uint32_t(i / sp.nb) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_m128(N);
    int ia = 0, ib = 0, n = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < sc.n_items; w += gridDim.x, ++n) {
      const Item it = item_at<N>(sc, w);
      // the epilogue has read the previous item's accumulators out
      if (!mbar_wait(acc_empty, (uint32_t(n) & 1u) ^ 1u) || *abort_p) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; ok && kb < a.n_kblk; ++kb) {
        const int sa = ia & 1;
        if (!mbar_wait(a_full(sa), uint32_t(ia >> 1) & 1u) || *abort_p) {
          ok = false;
          break;
        }
        const uint32_t xa = sA + sa * slot_a;
        for (int k = 0; k < a.K; ++k) {
          const int s = ib % sp.nb;
          if (!mbar_wait(b_full(s), uint32_t(ib / sp.nb) & 1u) || *abort_p) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int sh = sp.pad - (a.K - 1 - k) * a.dil;  // x slot row of the item's first token
          const uint64_t bd = sw128_desc(sB + s * kBStage);
          for (int h = 0; h < it.nh; ++h) {
            const uint64_t ad = sw128_desc(xa + uint32_t(128 * h + sh) * 128u);
#pragma unroll
            for (int j = 0; j < BK / UK; ++j)
              mma_bf16(tmem + uint32_t(h * N), ad + 2 * j, bd + 2 * j, idesc,
                       (kb > 0 || k > 0 || j > 0) ? 1u : 0u);
          }
          mma_commit(b_empty(s));
          ++ib;
        }
        if (!ok) break;
        mma_commit(a_empty(sa));
        ++ia;
      }
      if (ok) mma_commit(acc_full);
    }
    if (!ok && !*abort_p) fail();
    // every MMA issued above completes before the tensor memory is freed
    mma_commit(mma_done);
    if (!mbar_wait(mma_done, 0)) fail();
  } else if (warp >= 2) {
    // epilogue: warp w drains TMEM lanes 32 (w % 4) .. +31 of accumulator (w - 2) / 4
    const int e = warp - 2, q = warp & 3, h = e >> 2;
    uint8_t* const stage = generic(sStage) + e * kStageWarp;
    float* const bias_w = reinterpret_cast<float*>(generic(sBias)) + e * N;
    int n = 0;
    for (int w = blockIdx.x; w < sc.n_items; w += gridDim.x, ++n) {
      const Item it = item_at<N>(sc, w);
      // this warp's copy of the item's bias (zero past Cout or without one)
      __syncwarp();
      for (int i = lane; i < N; i += 32) {
        const int oc = it.n0 + i;
        float v = 0.0f;
        if (a.bias && oc < a.Cout)
          v = a.bias_f32 ? __ldg(static_cast<const float*>(a.bias) + int64_t(oc) * a.bias_s)
                         : bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.bias) + int64_t(oc) * a.bias_s));
        bias_w[i] = v;
      }
      __syncwarp();
      // lane 0 waits and tells the warp, so the warp-wide tcgen05.ld below is
      // reached by all lanes or by none
      int st = 0;
      if (lane == 0) {
        st = mbar_wait(acc_full, uint32_t(n) & 1u) ? (*abort_p ? 1 : 0) : 2;
        if (st == 2) fail();
      }
      st = __shfl_sync(0xffffffffu, st, 0);
      if (st) break;
      tc_fence_after();
      uint32_t pk[N / 2];  // the row as packed BF16
      if (h < it.nh) {
        const uint32_t taddr = tmem + (uint32_t(q * 32) << 16) + uint32_t(h * N);
#pragma unroll
        for (int c = 0; c < N; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + uint32_t(c), r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[c / 2 + j] = pack_bf16x2(__uint_as_float(r[2 * j]) + bias_w[c + 2 * j],
                                        __uint_as_float(r[2 * j + 1]) + bias_w[c + 2 * j + 1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);  // the accumulators may be overwritten
      if (h >= it.nh) continue;
      // rows t_row .. t_row + 31, kChunk columns per round through the staging
      // rows: each lane writes its row piece, then every store instruction
      // writes 8 whole row pieces of kChunk * 2 bytes
      const int t_row = it.t0 + h * 128 + q * 32;
      const int ncols = a.Cout - it.n0 < N ? a.Cout - it.n0 : N;  // a multiple of 8
      uint16_t* const obase = a.out + int64_t(it.bb) * a.o_sb + it.n0;
#pragma unroll
      for (int c = 0; c < N; c += kChunk) {
        if (c >= ncols) break;
        uint8_t* row = stage + lane * kStageRow;
#pragma unroll
        for (int p = 0; p < kChunk / 8; ++p)
          *reinterpret_cast<uint4*>(row + 16 * p) =
              make_uint4(pk[c / 2 + 4 * p], pk[c / 2 + 4 * p + 1], pk[c / 2 + 4 * p + 2],
                         pk[c / 2 + 4 * p + 3]);
        __syncwarp();
        constexpr int kPieces = kChunk / 8;        // 16-byte pieces per row piece
        constexpr int kRowsPerStore = 32 / kPieces;
#pragma unroll
        for (int i = 0; i < 32 / kRowsPerStore; ++i) {
          const int rr = i * kRowsPerStore + lane / kPieces, pc = lane % kPieces;
          const int t = t_row + rr, col = c + pc * 8;
          if (t < a.T && col < ncols)
            *reinterpret_cast<uint4*>(obase + int64_t(t) * a.o_st + col) =
                *reinterpret_cast<const uint4*>(stage + rr * kStageRow + pc * 16);
        }
        __syncwarp();
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// weight [Cout, Cin, K] (any strides, BF16 or FP32) -> packed [K, Cout, Cin] BF16
// (nearest-even for FP32); consecutive threads write consecutive input channels.
__global__ void pack_weight_kernel(const void* w, int w_f32, int64_t s_oc, int64_t s_ic, int64_t s_k,
                                   uint16_t* packed, int64_t Cout, int64_t Cin, int64_t K) {
  const int64_t n = K * Cout * Cin;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t ic = i % Cin, r = i / Cin, oc = r % Cout, k = r / Cout;
    const int64_t o = oc * s_oc + ic * s_ic + k * s_k;
    packed[i] = w_f32 ? f32_to_bf16(__ldg(static_cast<const float*>(w) + o))
                      : __ldg(static_cast<const uint16_t*>(w) + o);
  }
}

// ---- host side --------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A 3-D BF16 tensor map (innermost dimension contiguous) with a box of
// (64, box1, 1) elements and 128-byte swizzling; out-of-range elements read 0.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {uint32_t(BK), box1, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef CCC_FULLCONV_N
#define CCC_FULLCONV_N 256  // output channels per tile of the persistent kernel
#endif
constexpr int kSharedN = CCC_FULLCONV_N;
static_assert(kSharedN == 128 || kSharedN == 256, "N of the persistent kernel's tile");
constexpr size_t kMaxSmem = 232448;  // 227 KB: the per-block opt-in limit

ContextCache g_attr_done;
ContextCache g_sm_count;

cudaError_t smem_attributes() {
  long long done = 0;
  if (g_attr_done.get(&done) && done) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(fullconv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(fullconv_persistent_kernel<kSharedN>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(kMaxSmem));
  if (err == cudaSuccess) g_attr_done.put(1);
  return err;
}

cudaError_t sm_count(int* n) {
  long long v = 0;
  if (g_sm_count.get(&v) && v > 0) {
    *n = int(v);
    return cudaSuccess;
  }
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (err == cudaSuccess) g_sm_count.put(*n);
  return err;
}

// Persistent-kernel plan for this receptive field, or false when the x slots
// and at least two weight stages would not fit (then the per-tap kernel
// serves the call).
bool shared_plan(int64_t K, int64_t dil, SharedPlan& sp, size_t& smem) {
  const int64_t P = (K - 1) * dil;
  const int64_t padr = (P + 15) / 16 * 16;
  if (padr > 256) return false;
  sp.pad = int(padr);
  sp.ra = 256 + sp.pad;
  const size_t fixed = persistent_fixed_smem<kSharedN>(sp.ra);
  const size_t bstage = size_t(kSharedN) * BK * 2;
  if (fixed + 2 * bstage > kMaxSmem) return false;
  sp.nb = int(std::min<size_t>(8, (kMaxSmem - fixed) / bstage));
  smem = fixed + size_t(sp.nb) * bstage;
  return true;
}

// Whole tiles fill full waves of `grid_max` CTAs; when the rest would fill at
// most half a wave, it is cut into half tiles that all run in one last round.
Sched make_sched(int64_t T, int64_t Cout, int64_t B, int grid_max) {
  Sched sc{};
  sc.n_tb = int((T + 255) / 256);
  sc.n_ob = int((Cout + kSharedN - 1) / kSharedN);
  const int64_t n_tiles = int64_t(sc.n_tb) * sc.n_ob * B;
  const int64_t r = n_tiles % grid_max;
  if (r != 0 && 2 * r <= grid_max) {
    sc.n_main = int(n_tiles - r);
    sc.n_items = int(n_tiles + r);
  } else {
    sc.n_main = sc.n_items = int(n_tiles);
  }
  return sc;
}

}  // namespace fullconv

cudaError_t launch_fullconv(const FullConvArgs& f, cudaStream_t stream) {
  using namespace fullconv;
  const cudaError_t err = smem_attributes();
  if (err != cudaSuccess) return err;
  Args a{};
  a.out = f.out;
  a.o_sb = f.o_sb;
  a.o_st = f.o_st;
  a.bias = f.bias;
  a.bias_f32 = f.bias_f32;
  a.bias_s = f.bias_s;
  a.T = int(f.T);
  a.Cout = f.Cout;
  a.K = f.K;
  a.dil = f.dil;
  a.n_kblk = (f.Cin + BK - 1) / BK;
  a.status = f.status;
  // x: dims (Cin, T, B), row strides in bytes (the batch stride of a single
  // batch row is never used; any legal value serves); packed weight: dims
  // (Cin, Cout, K), contiguous
  const uint64_t xs_t = uint64_t(f.x_st) * 2;
  const uint64_t xs_b = f.B > 1 ? uint64_t(f.x_sb) * 2 : xs_t * uint64_t(f.T > 0 ? f.T : 1);
  const uint64_t ws_o = uint64_t(f.Cin) * 2, ws_k = ws_o * uint64_t(f.Cout);
  CUtensorMap mx, mw;
  SharedPlan sp{};
  size_t smem = 0;
  if (shared_plan(f.K, f.dil, sp, smem)) {
    if (!make_map(&mx, f.x, uint64_t(f.Cin), uint64_t(f.T), uint64_t(f.B), xs_t, xs_b,
                  uint32_t(sp.ra / 2)) ||
        !make_map(&mw, f.w, uint64_t(f.Cin), uint64_t(f.Cout), uint64_t(f.K), ws_o, ws_k, kSharedN))
      return cudaErrorInvalidValue;
    int nsm = 0;
    const cudaError_t e2 = sm_count(&nsm);
    if (e2 != cudaSuccess) return e2;
    const Sched sc = make_sched(f.T, f.Cout, f.B, nsm);
    const unsigned grid = unsigned(std::min(nsm, sc.n_items));
    return launch_kernel(fullconv_persistent_kernel<kSharedN>, dim3(grid), dim3(kPThreads), smem, stream,
                         true, mx, mw, a, sp, sc);
  }
  if (!make_map(&mx, f.x, uint64_t(f.Cin), uint64_t(f.T), uint64_t(f.B), xs_t, xs_b, BM) ||
      !make_map(&mw, f.w, uint64_t(f.Cin), uint64_t(f.Cout), uint64_t(f.K), ws_o, ws_k, BN))
    return cudaErrorInvalidValue;
  const dim3 grid(unsigned((f.T + BM - 1) / BM), unsigned((f.Cout + BN - 1) / BN), unsigned(f.B));
  return launch_kernel(fullconv_kernel, grid, dim3(kThreads), kSmemBytes, stream, true, mx, mw, a);
}

cudaError_t launch_pack_weight(const void* w, int w_f32, int64_t s_oc, int64_t s_ic, int64_t s_k,
                               uint16_t* packed, int64_t Cout, int64_t Cin, int64_t K,
                               cudaStream_t stream) {
  const int64_t n = K * Cout * Cin;
  const unsigned blocks = unsigned(std::min<int64_t>((n + 255) / 256, 152 * 8));
  fullconv::pack_weight_kernel<<<blocks, 256, 0, stream>>>(w, w_f32, s_oc, s_ic, s_k, packed, Cout,
                                                           Cin, K);
  return cudaGetLastError();
}

}  // namespace ccc
