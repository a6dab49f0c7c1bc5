/*
 * ccc_conv1d -- depthwise causal conv1d on BF16 activations, filter width W in
 * 2..4 (four is the page's optimized route).
 *
 * C ABI of the CUDA library (libccc_conv1d.so).  All tensor memory is owned by
 * the caller and the library allocates nothing.  Its only global state is a
 * cache of launch facts kept per (device, CUDA context) -- kernel attributes,
 * occupancy figures -- and the built-in scratch array of
 * ccc_conv1d_bwd_noalloc; every other call may run concurrently with others on
 * different streams (on disjoint outputs).
 *
 * The operation (cuDNN frontend docs, "Causal Conv1d" page):
 *
 *   out[b,d,t] = act(bias[d] + sum_{k<W} weight[d,k] * xe[b,d,t-(W-1)+k])
 *
 * where xe is x extended on the left by the W - 1 entries of initial_states
 * (zeros when none are given); index 0 of the state axis is the oldest entry.
 * Tap W - 1 multiplies the current token (POPCORNBENCH conv1d page, the reasoning
 * section's causal-padding derivation: tap k reads position t + k - (K-1)).
 * act is SiLU, p * sigmoid(p), or the identity.
 *
 * Tensors are passed as ccc_tensor descriptors: a data pointer, a dtype, the
 * number of dimensions, and shape/stride arrays with strides in ELEMENTS.
 * Unless stated otherwise a data pointer is a DEVICE pointer on the current
 * device, and every kernel runs on the given stream (NULL = legacy default
 * stream, following the frontend overview page's stream convention).
 *
 * Error behaviour.  Every argument check runs on the host before any work is
 * enqueued; on a non-CCC_OK return nothing has been written.  The only
 * device-side error is malformed cu_seqlens.  The cuDNN page executes a device
 * trap for it; this library instead has every thread block validate the
 * offsets, skip all of its writes and, when d_status is not NULL, record
 * CCC_ERR_BAD_CU_SEQLENS in *d_status (first error wins).  The CUDA context
 * stays usable; the outputs of that call are unspecified.  Read the word with
 * ccc_read_status.
 */
#ifndef CCC_CONV1D_H
#define CCC_CONV1D_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define CCC_CONV1D_ABI_VERSION 2
#define CCC_CONV1D_WIDTH 4

typedef enum {
    CCC_OK = 0,
    CCC_ERR_INVALID_ARG = 1,      /* NULL where required, bad shape/dtype/rank, unknown enum */
    CCC_ERR_UNSUPPORTED = 2,      /* well-formed but declined: width outside 2..4, FP32 weight with
                                     bias, strides this library does not read, B != 1 when packed */
    CCC_ERR_ALIAS = 3,            /* an output overlaps an input or another output */
    CCC_ERR_NONDETERMINISTIC = 4, /* deterministic backward requested with a bias */
    CCC_ERR_WORKSPACE = 5,        /* workspace NULL, too small or not 16-byte aligned */
    CCC_ERR_CUDA = 6,             /* a CUDA runtime call or launch failed */
    CCC_ERR_BAD_CU_SEQLENS = 7,   /* device-detected malformed cu_seqlens (via d_status) */
    CCC_ERR_SCRATCH_LIMIT = 8,    /* ccc_conv1d_bwd_noalloc: the problem needs more scratch
                                     than CCC_CONV1D_NOALLOC_SCRATCH_BYTES */
    CCC_ERR_DEVICE_TIMEOUT = 9    /* ccc_fullconv1d_fwd: a bounded wait on the device ran out
                                     (via d_status); the call's output is unspecified */
} ccc_status;

typedef enum { CCC_BF16 = 0, CCC_F32 = 1, CCC_I32 = 2 } ccc_dtype;

typedef enum { CCC_ACT_NONE = 0, CCC_ACT_SILU = 1 } ccc_act;

typedef struct {
    void *data;        /* device pointer (may be NULL only when numel == 0) */
    int32_t dtype;     /* ccc_dtype */
    int32_t ndim;      /* 1, 2 or 3 */
    int64_t shape[3];  /* entries past ndim are ignored */
    int64_t stride[3]; /* in elements */
} ccc_tensor;

/*
 * Forward (cuDNN "Causal Conv1d" page: the tensor list, the paragraph on
 * [B, T, D] storage passed as a transpose(1, 2) view, and the paragraph on the
 * optimized route: dense and cu_seqlens-packed, BF16 activations, width four,
 * W-1 initial and final state).
 *
 *   x               [B, D, T] BF16.  Two layouts are read in place:
 *                     channel-last: stride[1] == 1 (the transpose view of
 *                       [B, T, D] storage; stride[2] >= D);
 *                     time-contiguous: stride[2] == 1.
 *                   Any other layout returns CCC_ERR_UNSUPPORTED.
 *   weight          [D, W] BF16, W in 2..4 (the page's tensor list gives
 *                   weight[D, W]; its optimized route is W = 4), or FP32 only
 *                   when bias is NULL (the page declines FP32 weight with
 *                   bias); any strides.  Every state below is [S, D, W - 1].
 *   bias            [D] BF16 or NULL.
 *   cu_seqlens      [N + 1] int32 or NULL.  When given, x has B == 1 and holds
 *                   N sequences back to back along T; no tap reads across a
 *                   boundary.  Validated on the device (see above): offsets
 *                   start at 0, end at T, and strictly increase.
 *   seq_idx         [B, T] int32 or NULL, any non-negative strides: per-token
 *                   sequence ids (the page's seq_idx[B, T] keyword).  Tokens of
 *                   a row that carry the same id form one sequence: a tap of
 *                   token t reads a token of another id as zero.  The page makes
 *                   it mutually exclusive with cu_seqlens (both given:
 *                   CCC_ERR_INVALID_ARG); the page defines no state for it, so
 *                   initial_states or final_states with seq_idx return
 *                   CCC_ERR_UNSUPPORTED.
 *   initial_states  [S, D, W-1] BF16 contiguous or NULL; S = B (dense) or N (packed).
 *   out             [B, D, T] BF16, same layout kind as x (its own strides).
 *   final_states    [S, D, W-1] BF16 contiguous or NULL: xe[T-W+1 .. T-1] of
 *                   each sequence, a bitwise copy (initial-state entries when
 *                   T < W - 1).
 *                   Must not overlap x, weight, bias, cu_seqlens or
 *                   initial_states (CCC_ERR_ALIAS, the page's aliasing rule).
 *   activation      ccc_act.
 *   d_status        device int or NULL; see "Error behaviour".
 *
 * T == 0 is allowed (final_states then equals initial_states, or zeros).
 */
ccc_status ccc_conv1d_fwd(const ccc_tensor *x, const ccc_tensor *weight, const ccc_tensor *bias,
                          const ccc_tensor *cu_seqlens, const ccc_tensor *seq_idx,
                          const ccc_tensor *initial_states, const ccc_tensor *out,
                          const ccc_tensor *final_states, int activation, int *d_status,
                          cudaStream_t stream);

/*
 * Workspace bytes that ccc_conv1d_bwd needs for this x (shape and layout) and
 * mode, on the current device.  Returns 0 for an x that ccc_conv1d_bwd would
 * reject.  The value depends on the device's SM count, so query it on the
 * device you launch on.
 */
size_t ccc_conv1d_bwd_workspace_size(const ccc_tensor *x, int deterministic);

/*
 * Backward (cuDNN "Causal Conv1d" page: forward and backward on the optimized
 * route; the paragraph on determinism).  The pre-activation is recomputed
 * from x; nothing from the forward is needed.
 *
 *   x, weight, bias, cu_seqlens, seq_idx, initial_states   as in ccc_conv1d_fwd
 *                   (with seq_idx, dfinal_states and dinitial_states must be NULL).
 *   dout            [B, D, T] BF16, same layout kind as x: dL/dout.
 *   dfinal_states   [S, D, W-1] BF16 contiguous or NULL (NULL = zero gradient).
 *   dx              [B, D, T] BF16, same layout kind as x.
 *   dweight         [D, W], dtype of weight, any strides.
 *   dbias           [D] BF16; required when bias is given, else must be NULL.
 *   dinitial_states [S, D, W-1] BF16 contiguous or NULL (allowed only with
 *                   initial_states).
 *   deterministic   0 or 1.  The page's rule is kept: 1 (the deterministic
 *                   route) is declined for calls with a bias
 *                   (CCC_ERR_NONDETERMINISTIC).  This library computes both
 *                   modes the same way -- unique FP32 per-block partial sums
 *                   followed by a fixed-order reduction -- so dweight/dbias
 *                   are bitwise reproducible in either.
 *   workspace       device buffer of at least
 *                   ccc_conv1d_bwd_workspace_size(x, deterministic) bytes,
 *                   16-byte aligned; contents on entry are ignored.
 *
 * Outputs must not overlap each other or any input (CCC_ERR_ALIAS).
 */
ccc_status ccc_conv1d_bwd(const ccc_tensor *x, const ccc_tensor *weight, const ccc_tensor *bias,
                          const ccc_tensor *cu_seqlens, const ccc_tensor *seq_idx,
                          const ccc_tensor *initial_states, const ccc_tensor *dout,
                          const ccc_tensor *dfinal_states, const ccc_tensor *dx,
                          const ccc_tensor *dweight, const ccc_tensor *dbias,
                          const ccc_tensor *dinitial_states, int activation, int deterministic,
                          void *workspace, size_t workspace_bytes, int *d_status,
                          cudaStream_t stream);

/*
 * Backward without any allocation -- no counterpart in the pages; it exists for
 * callers that cannot allocate device memory.  Such callers are programs
 * embedded in a host that owns all device memory and forbids allocation while
 * it runs (a server with a fixed memory budget, a plugin interface that hands
 * over only the operation's own tensors): they cannot provide the workspace
 * ccc_conv1d_bwd asks for.
 *
 * Same arguments and results as ccc_conv1d_bwd without seq_idx (it takes no
 * per-token sequence ids), minus the workspace: the FP32
 * sums live in a scratch array of CCC_CONV1D_NOALLOC_SCRATCH_BYTES built into
 * the library, present in device memory on every GPU that loads it, until the
 * library is unloaded.  Nothing is allocated (no cudaMalloc, no cudaFree, no
 * allocating library routine).
 *
 *   - The first call in a CUDA context (normally the device's primary
 *     context), with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress); make that first call before any stream
 *     capture.  A new context on the same device (after cudaDeviceReset, for
 *     example) gets its own lookup on its first call.
 *   - A problem whose workspace (ccc_conv1d_bwd_workspace_size) exceeds the
 *     scratch returns CCC_ERR_SCRATCH_LIMIT and enqueues nothing.
 *   - All calls on a device share the array.  Calls whose work overlaps on
 *     the GPU (different streams at once) race on it; calls on one stream are
 *     ordered.  Each call zeroes or overwrites what it reads, so an earlier
 *     call's contents never leak into a result.
 */
#define CCC_CONV1D_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

ccc_status ccc_conv1d_bwd_noalloc(const ccc_tensor *x, const ccc_tensor *weight,
                                  const ccc_tensor *bias, const ccc_tensor *cu_seqlens,
                                  const ccc_tensor *initial_states, const ccc_tensor *dout,
                                  const ccc_tensor *dfinal_states, const ccc_tensor *dx,
                                  const ccc_tensor *dweight, const ccc_tensor *dbias,
                                  const ccc_tensor *dinitial_states, int activation,
                                  int deterministic, int *d_status, cudaStream_t stream);

/*
 * Decode update (cuDNN "Causal Conv1d" page, the paragraph on passing
 * final_states to causal_conv1d_update, which mutates that state in place;
 * the page's "commonly consumed causal-conv1d interface" also takes several
 * new tokens per row).
 *
 *   x           [B, D] BF16 (one token per row) or [B, D, L] BF16 (L >= 0 tokens
 *               per row, any token stride), stride[1] == 1.
 *   conv_state  [B, D, W-1] BF16 contiguous, read and overwritten in place: after
 *               each token, [s1 .. s(W-2), x] (bitwise): the layout final_states
 *               uses.
 *   weight      [D, W] as in ccc_conv1d_fwd;  bias [D] BF16 or NULL.
 *   out         shaped like x, stride[1] == 1; for each token in order:
 *               act(bias + sum_{k<W-1} w_k*s_k + w_(W-1)*x).
 *
 * The result equals ccc_conv1d_fwd over the L tokens with conv_state as the
 * initial state and the new state as the final state, bitwise.  L == 0 (or
 * B == 0) computes nothing and leaves the state unchanged.  out may be x itself
 * (same pointer, shape and strides: the update is then in place) but must not
 * otherwise overlap it; out must not overlap conv_state, weight or bias, and x
 * must not overlap conv_state (CCC_ERR_ALIAS).
 */
ccc_status ccc_conv1d_update(const ccc_tensor *x, const ccc_tensor *conv_state,
                             const ccc_tensor *weight, const ccc_tensor *bias,
                             const ccc_tensor *out, int activation, cudaStream_t stream);

/*
 * Full-channel dilated causal conv1d (POPCORNBENCH conv1d page: a Conv1d over
 * all input channels with dilation, left-padded by P = (K-1)*dilation; the
 * reasoning section derives that tap k reads input position t + k*dilation - P
 * and the listing adds an optional bias):
 *
 *   out[b,oc,t] = bias[oc] + sum_{ic<Cin} sum_{k<K} W[oc,ic,k] * x[b,ic,t + k*dilation - P]
 *
 * with x read as zero at negative positions.  A dense contraction over input
 * channels and taps, computed on the tensor cores: BF16 operands, FP32
 * accumulation, BF16 output (rounded to nearest even).  Forward only.
 *
 * ccc_fullconv1d_pack_weight copies W into the tap-major layout the kernel
 * reads (do it once per weight update; the weight is not read otherwise):
 *
 *   weight   [Cout, Cin, K] BF16 or FP32 (rounded to BF16), any strides.
 *   packed   [K, Cout, Cin] BF16, contiguous; packed[k, oc, ic] = W[oc, ic, k].
 *            Must not overlap weight (CCC_ERR_ALIAS).
 *
 * ccc_fullconv1d_fwd:
 *
 *   x              [B, Cin, T] BF16, channel-last: stride[1] == 1 (the
 *                  transpose view of [B, T, Cin] storage); the token and batch
 *                  strides multiples of 8 elements, data 16-byte aligned,
 *                  Cin a multiple of 8.  Other layouts: CCC_ERR_UNSUPPORTED.
 *   packed_weight  [K, Cout, Cin] BF16 from ccc_fullconv1d_pack_weight
 *                  (contiguous, 16-byte aligned); Cout a multiple of 8.
 *   bias           [Cout] BF16 or FP32 (added in FP32), any stride, or NULL.
 *   dilation       >= 1.
 *   out            [B, Cout, T] BF16, channel-last like x (same rules).
 *                  Must not overlap x, packed_weight or bias (CCC_ERR_ALIAS).
 *   d_status       device int or NULL: a wait inside the kernel that runs out
 *                  (it cannot in a working GPU) records CCC_ERR_DEVICE_TIMEOUT.
 *
 * B == 0 or T == 0 computes nothing.  Limits (else CCC_ERR_UNSUPPORTED): B and
 * ceil(Cout / 256) at most 65535, K at most 1024, (K-1)*dilation and T below
 * 2^30, B * ceil(T / 256) * ceil(Cout / 256) below 2^30.
 *
 * The call launches one CTA per SM (receptive field (K-1)*dilation up to 256
 * tokens; longer ones take one CTA per tile of 128 tokens x 256 channels), so
 * it occupies the whole GPU while it runs.
 */
ccc_status ccc_fullconv1d_pack_weight(const ccc_tensor *weight, const ccc_tensor *packed,
                                      cudaStream_t stream);

ccc_status ccc_fullconv1d_fwd(const ccc_tensor *x, const ccc_tensor *packed_weight,
                              const ccc_tensor *bias, int dilation, const ccc_tensor *out,
                              int *d_status, cudaStream_t stream);

/*
 * Synchronise `stream`, read the device status word written by the kernels
 * (d_status, a device pointer), reset it to 0, and return it as a ccc_status
 * (CCC_OK when no error was recorded).  Returns CCC_ERR_CUDA if the
 * synchronisation or copy fails.
 */
ccc_status ccc_read_status(int *d_status, cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *ccc_status_string(int status);

/* CCC_CONV1D_ABI_VERSION of the built library. */
int ccc_conv1d_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCC_CONV1D_H */
