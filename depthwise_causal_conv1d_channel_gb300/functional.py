"""Model-facing operations: causal_conv1d (with autograd) and causal_conv1d_update.

The argument lists follow the cuDNN frontend "Causal Conv1d" page (the
commonly consumed causal-conv1d interface): x [B, D, T] -- or the
transpose(1, 2) view of [B, T, D] storage, read in place --, weight [D, 4],
optional bias [D], optional per-token sequence ids seq_idx [B, T], optional
packed cu_seqlens [N + 1] (mutually exclusive with seq_idx), optional
initial_states and returned final_states of width W - 1 = 3, and a SiLU
activation.  Every step runs in the CUDA library through
the C ABI; this module allocates outputs, picks the determinism mode and maps
status codes to Python exceptions.
"""

from __future__ import annotations

import os
import warnings
from typing import Optional

import torch

from . import _abi

_ACTIVATIONS = {"silu": _abi.CCC_ACT_SILU, "swish": _abi.CCC_ACT_SILU, None: _abi.CCC_ACT_NONE,
                "identity": _abi.CCC_ACT_NONE, "none": _abi.CCC_ACT_NONE}

_status_words = {}


def _activation_code(activation) -> int:
    if activation not in _ACTIVATIONS:
        raise ValueError(f"activation must be 'silu' or None, got {activation!r}")
    return _ACTIVATIONS[activation]


def status_word(device: torch.device) -> torch.Tensor:
    """The per-device int32 status word every call of this module passes to the
    kernels (malformed cu_seqlens are reported there instead of a device trap)."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    w = _status_words.get(idx)
    if w is None:
        w = torch.zeros(1, dtype=torch.int32, device=torch.device("cuda", idx))
        _status_words[idx] = w
    return w


def check_status(device=None, stream=None) -> None:
    """Synchronise and raise if a kernel recorded a device-side error since the
    last check (for example malformed cu_seqlens); clears the word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = _abi.ccc_read_status(status_word(dev), stream or torch.cuda.current_stream(dev))
    if st != _abi.CCC_OK:
        raise _abi.Conv1dError(st, "device status")


def _raise(st: int, where: str):
    if st == _abi.CCC_OK:
        return
    if st == _abi.CCC_ERR_ALIAS:
        raise ValueError(f"{where}: {_abi.status_string(st)}")
    if st == _abi.CCC_ERR_INVALID_ARG:
        raise ValueError(f"{where}: {_abi.status_string(st)}")
    if st == _abi.CCC_ERR_UNSUPPORTED:
        raise NotImplementedError(f"{where}: {_abi.status_string(st)}")
    raise _abi.Conv1dError(st, where)


def _debug_check(device):
    if os.environ.get("CCC_CONV1D_CHECK_STATUS", "0") not in ("", "0"):
        check_status(device)


def _like_x(t: torch.Tensor, x: torch.Tensor) -> torch.Tensor:
    """t laid out like x (same strides), copying only when the layouts differ."""
    if t.stride() == x.stride():
        return t
    out = torch.empty_strided(x.shape, x.stride(), dtype=t.dtype, device=t.device)
    out.copy_(t)
    return out


def _deterministic_mode(has_bias: bool, deterministic: Optional[bool]) -> bool:
    """The cuDNN page's rule: torch.use_deterministic_algorithms selects the
    deterministic dweight route for bias-free calls; with a bias there is none,
    so raise RuntimeError, or warn and take the default route under
    warn_only=True.  A per-call deterministic=True/False overrides the global
    setting.  (The kernels compute both routes as fixed-order sums of per-block
    partials, so the default route is bitwise repeatable too.)"""
    want = torch.are_deterministic_algorithms_enabled() if deterministic is None else deterministic
    if not want:
        return False
    if not has_bias:
        return True
    msg = "causal_conv1d backward with bias has no deterministic dbias route"
    if deterministic is None and torch.is_deterministic_algorithms_warn_only_enabled():
        warnings.warn(msg)
        return False
    raise RuntimeError(msg)


class _CausalConv1dFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, cu_seqlens, seq_idx, initial_states, final_states_out,
                want_final, act, deterministic):
        out = torch.empty_like(x)  # same strides as x: channel-last in, channel-last out
        S = x.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
        final = None
        if want_final:
            final = final_states_out if final_states_out is not None else torch.empty(
                (S, x.shape[1], weight.shape[1] - 1), dtype=x.dtype, device=x.device)
        st = _abi.ccc_conv1d_fwd(x, weight, bias, cu_seqlens, initial_states, out, final, act,
                                 status_word(x.device), torch.cuda.current_stream(x.device),
                                 seq_idx=seq_idx)
        _raise(st, "causal_conv1d")
        _debug_check(x.device)
        ctx.save_for_backward(x, weight, bias, cu_seqlens, seq_idx, initial_states)
        ctx.act = act
        ctx.deterministic = deterministic
        if final_states_out is not None:
            ctx.mark_dirty(final_states_out)
        return out, final

    @staticmethod
    def backward(ctx, dout, dfinal):
        x, weight, bias, cu_seqlens, seq_idx, initial_states = ctx.saved_tensors
        det = _deterministic_mode(bias is not None, ctx.deterministic)
        if dout is None:
            dout = torch.zeros_like(x)
        dout = _like_x(dout, x)
        if dfinal is not None:
            dfinal = dfinal.contiguous()
        dx = torch.empty_like(x)
        dweight = torch.empty_like(weight, memory_format=torch.contiguous_format)
        dbias = torch.empty_like(bias) if bias is not None else None
        dinit = None
        if initial_states is not None and ctx.needs_input_grad[5]:
            dinit = torch.empty_like(initial_states)
        ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(x, det), dtype=torch.uint8,
                         device=x.device)
        st = _abi.ccc_conv1d_bwd(x, weight, bias, cu_seqlens, initial_states, dout, dfinal, dx,
                                 dweight, dbias, dinit, ctx.act, det, ws, status_word(x.device),
                                 torch.cuda.current_stream(x.device), seq_idx=seq_idx)
        _raise(st, "causal_conv1d backward")
        _debug_check(x.device)
        return dx, dweight, dbias, None, None, dinit, None, None, None, None


def causal_conv1d(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
                  seq_idx: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                  initial_states: Optional[torch.Tensor] = None, return_final_states: bool = False,
                  final_states_out: Optional[torch.Tensor] = None, activation: Optional[str] = "silu",
                  deterministic: Optional[bool] = None):
    """Depthwise causal conv1d of width W = weight.shape[1] (2..4; four is the
    page's optimized route), BF16 activations.

    out[b, d, t] = act(bias[d] + sum_k weight[d, k] * xe[b, d, t - (W-1) + k]) where
    xe is x preceded by the W - 1 initial-state entries (zeros when none);
    initial_states and final_states are [B or N, D, W - 1].

    ``seq_idx`` [B, T] int32 gives every token a sequence id: tokens of a row
    with the same id form one sequence, and a tap reads a token of another id as
    zero.  It excludes cu_seqlens (ValueError) and has no initial or final
    state (NotImplementedError).

    Returns ``out`` (same shape and strides as x) or ``(out, final_states)`` when
    ``return_final_states`` is set or ``final_states_out`` is given.  Differentiable
    in x, weight, bias and initial_states.  ``deterministic`` (default: follow
    ``torch.use_deterministic_algorithms``) selects the reproducible dweight route.
    """
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    if seq_idx is not None:
        if seq_idx.dtype != torch.int32:
            raise ValueError("seq_idx must be int32")
        if cu_seqlens is not None:
            raise ValueError("seq_idx and cu_seqlens are mutually exclusive")
        if initial_states is not None or return_final_states or final_states_out is not None:
            raise NotImplementedError("seq_idx defines no initial or final state")
    act = _activation_code(activation)
    want_final = bool(return_final_states) or final_states_out is not None
    out, final = _CausalConv1dFn.apply(x, weight, bias, cu_seqlens, seq_idx, initial_states,
                                       final_states_out, want_final, act, deterministic)
    return (out, final) if want_final else out


def causal_conv1d_update(x: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
                         bias: Optional[torch.Tensor] = None, activation: Optional[str] = "silu",
                         out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode step(s): x [B, D] is the new token, or x [B, D, L] the next L
    tokens of every row; conv_state [B, D, W - 1] (the layout final_states uses) is
    read and mutated in place, token by token, to the last three extended
    inputs.  Returns out shaped like x.  The kernels read each token's D
    channels contiguously: a [B, D, L] x whose channel stride is not 1 is
    restrided first (a copy), and a new out is allocated with channel stride 1
    ([B, L, D] storage seen as [B, D, L])."""
    act = _activation_code(activation)
    if x.dim() == 3 and x.shape[1] > 1 and x.stride(1) != 1:
        x = x.transpose(1, 2).contiguous().transpose(1, 2)
    if out is None:
        if x.dim() == 3:
            out = torch.empty(x.shape[0], x.shape[2], x.shape[1], dtype=x.dtype,
                              device=x.device).transpose(1, 2)
        else:
            out = torch.empty_like(x, memory_format=torch.contiguous_format)
    st = _abi.ccc_conv1d_update(x, conv_state, weight, bias, out, act,
                                torch.cuda.current_stream(x.device))
    _raise(st, "causal_conv1d_update")
    return out


def pack_full_conv_weight(weight: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The full-channel conv's weight [Cout, Cin, K] (BF16, or FP32 rounded to
    BF16) copied tap-major into the [K, Cout, Cin] BF16 layout that
    full_causal_conv1d's kernel reads; pack once per weight update."""
    K, Cout, Cin = weight.shape[2], weight.shape[0], weight.shape[1]
    if out is None:
        out = torch.empty(K, Cout, Cin, dtype=torch.bfloat16, device=weight.device)
    st = _abi.ccc_fullconv1d_pack_weight(weight, out, torch.cuda.current_stream(weight.device))
    _raise(st, "pack_full_conv_weight")
    return out


def full_causal_conv1d(x: torch.Tensor, weight: Optional[torch.Tensor] = None,
                       bias: Optional[torch.Tensor] = None, dilation: int = 1,
                       packed_weight: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Full-channel dilated causal conv1d (the POPCORNBENCH conv1d page's
    operation), forward only:

        out[b, oc, t] = bias[oc] + sum_{ic, k} weight[oc, ic, k] * x[b, ic, t + k*dilation - P]

    with P = (K - 1) * dilation and x read as zero before position 0.  x is
    [B, Cin, T] BF16; the kernel reads channel-last storage ([B, T, Cin] seen
    as its transpose), so another layout is restrided first (a copy).  Pass
    ``weight`` [Cout, Cin, K] or its ``packed_weight`` from
    pack_full_conv_weight.  Returns out [B, Cout, T] BF16 with channel-last
    storage.  Runs on the tensor cores (BF16 operands, FP32 accumulation)."""
    if torch.is_grad_enabled() and (x.requires_grad or (weight is not None and weight.requires_grad)
                                    or (bias is not None and bias.requires_grad)):
        raise NotImplementedError("full_causal_conv1d is forward only")
    if packed_weight is None:
        if weight is None:
            raise ValueError("pass weight or packed_weight")
        packed_weight = pack_full_conv_weight(weight)
    if x.dim() == 3 and x.shape[1] > 1 and x.stride(1) != 1:
        x = x.transpose(1, 2).contiguous().transpose(1, 2)
    B, T = x.shape[0], x.shape[2]
    Cout = packed_weight.shape[1]
    out = torch.empty(B, T, Cout, dtype=torch.bfloat16, device=x.device).transpose(1, 2)
    st = _abi.ccc_fullconv1d_fwd(x, packed_weight, bias, int(dilation), out, status_word(x.device),
                                 torch.cuda.current_stream(x.device))
    _raise(st, "full_causal_conv1d")
    _debug_check(x.device)
    return out
