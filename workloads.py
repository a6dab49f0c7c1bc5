"""Seeded synthetic inputs for the depthwise causal conv1d.

This module holds input generation only -- none of the operation's arithmetic.
It is the one piece of code that both the CUDA path's callers and the CPU
oracle's callers share, so that both sides see byte-identical inputs.

Recipe (every tensor): draw with ``torch.Generator().manual_seed(seed)`` on the
CPU, in the order the workload lists its tensors, in float32, then round to
bfloat16 (round-to-nearest-even) unless the tensor is float32 by definition.
``N(0,1)`` is ``torch.randn``; ``U(a,b)`` is ``a + (b-a) * torch.rand``.
"Channel-last" storage means the tensor is allocated ``[B, T, D]`` and handed
to the operation as its ``transpose(1, 2)`` view of logical shape ``[B, D, T]``
(the cuDNN "Causal Conv1d" page, paragraph on models that own ``[B, T, D]``
storage).

The five named workloads follow the shapes, dtypes and distributions of the
task's benchmark configurations; the packed workload's sequence lengths are
drawn with ``torch.randint(1, 4097, (16,))`` from the same generator, before
any tensor.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

BF16 = torch.bfloat16


def _normal(gen, shape):
    return torch.randn(shape, generator=gen, dtype=torch.float32)


def _uniform(gen, shape, lo, hi):
    return lo + (hi - lo) * torch.rand(shape, generator=gen, dtype=torch.float32)


@dataclasses.dataclass
class ConvInputs:
    """One call's inputs (CPU tensors).  ``x``/``g`` are logical [B, D, T] views."""

    x: torch.Tensor
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    initial_states: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    g: Optional[torch.Tensor]
    dfinal_states: Optional[torch.Tensor]
    activation: Optional[str]
    channel_last: bool
    deterministic: bool = False

    @property
    def n_seq(self) -> int:
        return self.x.shape[0] if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    @property
    def tokens(self) -> int:
        return self.x.shape[0] * self.x.shape[2]

    def to(self, device) -> "ConvInputs":
        def mv(t):
            if t is None:
                return None
            if self.channel_last and t.dim() == 3 and t is not self.initial_states and t is not self.dfinal_states:
                # keep the [B, T, D] storage behind the [B, D, T] view
                return t.transpose(1, 2).contiguous().to(device).transpose(1, 2)
            return t.to(device)

        return dataclasses.replace(
            self,
            x=mv(self.x), weight=mv(self.weight), bias=mv(self.bias),
            initial_states=mv(self.initial_states), cu_seqlens=mv(self.cu_seqlens),
            g=mv(self.g), dfinal_states=mv(self.dfinal_states),
        )


def make_inputs(B: int, D: int, T: int, *, channel_last: bool = True, seed: int = 0,
                weight_dtype=BF16, bias: bool = True, initial_states: bool = False,
                grad: bool = False, dfinal_states: bool = False, lengths=None,
                activation: Optional[str] = "silu", deterministic: bool = False,
                x_scale: float = 1.0, width: int = 4) -> ConvInputs:
    """Inputs of one call.  ``lengths`` (list of ints) makes a packed call:
    B must be 1 and T == sum(lengths).  ``width`` is the filter width W (weight
    [D, W], states [., D, W - 1]).  Draw order: x, weight, bias,
    initial_states, g, dfinal_states."""
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is not None:
        if B != 1 or int(sum(lengths)) != T:
            raise ValueError("packed inputs take B == 1 and T == sum(lengths)")
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    n_seq = B if cu is None else cu.numel() - 1

    def act_tensor():
        if channel_last:
            return (_normal(gen, (B, T, D)) * x_scale).to(BF16).transpose(1, 2)
        return (_normal(gen, (B, D, T)) * x_scale).to(BF16)

    x = act_tensor()
    w = _uniform(gen, (D, width), -0.5, 0.5)
    w = w if weight_dtype == torch.float32 else w.to(BF16)
    b = _uniform(gen, (D,), -0.1, 0.1).to(BF16) if bias else None
    init = _normal(gen, (n_seq, D, width - 1)).to(BF16) if initial_states else None
    g = act_tensor() if grad else None
    gf = _normal(gen, (n_seq, D, width - 1)).to(BF16) if dfinal_states else None
    return ConvInputs(x=x, weight=w, bias=b, initial_states=init, cu_seqlens=cu, g=g,
                      dfinal_states=gf, activation=activation, channel_last=channel_last,
                      deterministic=deterministic)


def packed_lengths(seed: int = 0, n_seq: int = 16, max_len: int = 4096):
    """Sequence lengths of the packed workload: U[1, max_len] integers, drawn
    first from the workload's generator."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(1, max_len + 1, (n_seq,), generator=gen).tolist(), gen


# ---- the five named workloads ------------------------------------------------

def dense_small(seed: int = 0) -> ConvInputs:
    """Forward only, dense: x [2, 64, 128] contiguous, BF16 weight and bias, no state."""
    return make_inputs(2, 64, 128, channel_last=False, seed=seed)


def dense_state(seed: int = 0) -> ConvInputs:
    """Dense forward+backward with state: x stored [4, 2048, 1536] channel-last,
    BF16 weight/bias, initial_states [4, 1536, 3], return final_states, grad_out."""
    return make_inputs(4, 1536, 2048, seed=seed, initial_states=True, grad=True)


def packed_varlen(seed: int = 0) -> ConvInputs:
    """Packed varlen forward+backward: 16 sequences of U[1, 4096] tokens, D = 2048,
    channel-last, FP32 weight, no bias, per-sequence initial states,
    deterministic weight gradient."""
    lengths, gen = packed_lengths(seed)
    T = int(sum(lengths))
    D = 2048
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths), 0).to(torch.int32)
    x = _normal(gen, (1, T, D)).to(BF16).transpose(1, 2)
    w = _uniform(gen, (D, 4), -0.5, 0.5)
    init = _normal(gen, (len(lengths), D, 3)).to(BF16)
    g = _normal(gen, (1, T, D)).to(BF16).transpose(1, 2)
    return ConvInputs(x=x, weight=w, bias=None, initial_states=init, cu_seqlens=cu, g=g,
                      dfinal_states=None, activation="silu", channel_last=True,
                      deterministic=True)


@dataclasses.dataclass
class UpdateInputs:
    conv_state: torch.Tensor   # [B, D, 3]
    x_seq: torch.Tensor        # [steps, B, D]
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    activation: Optional[str] = "silu"


def decode_update(seed: int = 0, B: int = 256, D: int = 4096, steps: int = 1000) -> UpdateInputs:
    """Decode update: state [256, 4096, 3], one token x [256, 4096] per step for
    ``steps`` chained steps, BF16 weight and bias."""
    gen = torch.Generator().manual_seed(seed)
    state = _normal(gen, (B, D, 3)).to(BF16)
    x_seq = _normal(gen, (steps, B, D)).to(BF16)
    w = _uniform(gen, (D, 4), -0.5, 0.5).to(BF16)
    b = _uniform(gen, (D,), -0.1, 0.1).to(BF16)
    return UpdateInputs(conv_state=state, x_seq=x_seq, weight=w, bias=b)


def dense_large(seed: int = 0, bias: bool = True) -> ConvInputs:
    """Large dense forward+backward: x stored [8, 8192, 5120] channel-last, BF16
    weight; with bias (atomic weight gradient) or bias-free (deterministic)."""
    return make_inputs(8, 5120, 8192, seed=seed, bias=bias, initial_states=True, grad=True,
                       deterministic=not bias)


WORKLOADS = {
    "dense_small": dense_small,
    "dense_state": dense_state,
    "packed_varlen": packed_varlen,
    "decode_update": decode_update,
    "dense_large": dense_large,
}


# ---- marshalling helpers (bit patterns, no arithmetic) ----------------------

def device_activations(B: int, D: int, T: int, device, seed: int, channel_last: bool = True):
    """A seeded N(0, 1) BF16 activation tensor drawn on the device, for sizes
    too large to draw on the host: [B, T, D] storage seen as its [B, D, T]
    transpose when ``channel_last``, else contiguous [B, D, T]."""
    gen = torch.Generator(device=device).manual_seed(seed)
    shape = (B, T, D) if channel_last else (B, D, T)
    t = torch.randn(shape, generator=gen, device=device, dtype=BF16)
    return t.transpose(1, 2) if channel_last else t


def bits(t: Optional[torch.Tensor]):
    """BF16 tensor -> numpy uint16 bit patterns (logical shape kept); float32 and
    int32 tensors are returned as numpy arrays of their own dtype."""
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == BF16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> BF16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(BF16)


def seq_ids(B: int, T: int, seed: int, kind: str = "runs", max_run: int = 64,
            n_ids: int = 3) -> torch.Tensor:
    """Per-token sequence ids [B, T] int32 (the seq_idx keyword of the cuDNN page).

    ``runs``: every row is cut into consecutive runs of U[1, max_run] tokens,
    numbered upward from a per-row offset (the usual packed-in-a-row layout);
    ``random``: every token draws an id from U{0, .., n_ids - 1}, so equal ids
    need not be adjacent."""
    gen = torch.Generator().manual_seed(seed)
    if kind == "random":
        return torch.randint(0, n_ids, (B, T), generator=gen, dtype=torch.int32)
    if kind != "runs":
        raise ValueError(f"unknown id layout {kind!r}")
    ids = torch.empty(B, T, dtype=torch.int32)
    for b in range(B):
        t, cur = 0, int(torch.randint(-100, 100, (1,), generator=gen))
        while t < T:
            n = int(torch.randint(1, max_run + 1, (1,), generator=gen))
            ids[b, t:t + n] = cur
            t += n
            cur += 1
    return ids


# ---- full-channel dilated causal conv1d (POPCORNBENCH conv1d page) -------------

@dataclasses.dataclass
class FullConvInputs:
    x: torch.Tensor                 # [B, Cin, T] BF16 (channel-last storage: [B, T, Cin])
    weight: torch.Tensor            # [Cout, Cin, K] BF16 or FP32
    bias: Optional[torch.Tensor]    # [Cout] BF16 or FP32, or None
    dilation: int

    def to(self, device) -> "FullConvInputs":
        return dataclasses.replace(
            self, x=self.x.transpose(1, 2).contiguous().to(device).transpose(1, 2),
            weight=self.weight.to(device), bias=None if self.bias is None else self.bias.to(device))


def fullconv_inputs(B: int, Cin: int, Cout: int, T: int, K: int, dilation: int, seed: int = 0,
                    bias: bool = True, weight_dtype=BF16, bias_dtype=BF16) -> FullConvInputs:
    """x ~ N(0, 1) stored [B, T, Cin]; weight and bias ~ U(-1/sqrt(Cin*K), +1/sqrt(Cin*K))
    (the bound of the page's listing's initialisation, fan-in Cin*K).  Draw
    order: x, weight, bias."""
    gen = torch.Generator().manual_seed(seed)
    x = _normal(gen, (B, T, Cin)).to(BF16).transpose(1, 2)
    bound = 1.0 / float(Cin * K) ** 0.5
    w = _uniform(gen, (Cout, Cin, K), -bound, bound)
    w = w if weight_dtype == torch.float32 else w.to(BF16)
    b = None
    if bias:
        b = _uniform(gen, (Cout,), -bound, bound)
        b = b if bias_dtype == torch.float32 else b.to(BF16)
    return FullConvInputs(x=x, weight=w, bias=b, dilation=dilation)


def fullconv_dilated(seed: int = 0) -> FullConvInputs:
    """The full-channel workload measured here: B = 8 rows of T = 4096 tokens,
    Cin = Cout = 1024, kernel size 4, dilation 2, BF16 bias (the page prints no
    sizes; this is a mid-size dilated causal layer)."""
    return fullconv_inputs(8, 1024, 1024, 4096, 4, 2, seed=seed)
