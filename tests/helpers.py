"""Shared test helpers: run the CUDA path and the oracle on the same seeded
inputs and compare with the tolerances the benchmark spec fixes.

Tolerances (stated once, used everywhere):
* final_states, update state: bit-exact.
* BF16 activations and gradients (out, dx, dinitial_states):
  |gpu - ref| <= 1e-2 + 1.6e-2 * |ref|, ref = the oracle's result rounded to BF16.
* dweight / dbias: |gpu - ref64| <= 1e-3 * sum|terms| (+ 2^-8 * |ref64| when the
  output is BF16: one BF16 rounding of the result, which the relative bound on
  the sum cannot absorb when the terms do not cancel).
* full-channel conv output: the same form, |gpu - ref64| <= 1e-3 * sum|terms| +
  2^-8 * |ref64|: the operands are BF16 (their products exact in FP32), the
  tensor cores accumulate Cin * K products in FP32 in an order of their own,
  and the result is rounded once to BF16.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import bits

ATOL = 1e-2
RTOL = 1.6e-2
WG_REL = 1e-3
BF16_HALF_ULP_REL = 2.0 ** -8


def decode(a):
    return oracle.bf16_decode(a)


def assert_bf16_close(gpu_bits, ref_bits, what=""):
    g = decode(gpu_bits)
    r = decode(ref_bits)
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu={g[i]} ref={r[i]}")


def assert_bits_equal(gpu_bits, ref_bits, what=""):
    if not np.array_equal(gpu_bits, ref_bits):
        n = int((gpu_bits != ref_bits).sum())
        i = np.argwhere(gpu_bits != ref_bits)[0]
        raise AssertionError(f"{what}: {n} elements differ bitwise; first at {tuple(i)}: "
                             f"gpu={gpu_bits[tuple(i)]:#06x} ref={ref_bits[tuple(i)]:#06x}")


def assert_wgrad_close(gpu_vals, ref64, abs_sum, bf16_out: bool, what=""):
    err = np.abs(gpu_vals - ref64)
    bound = WG_REL * abs_sum + (BF16_HALF_ULP_REL * np.abs(ref64) if bf16_out else 0.0)
    bound = bound + 1e-30
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst at {i}: "
                             f"gpu={gpu_vals[i]} ref={ref64[i]} sum|terms|={abs_sum[i]}")


def tensor_values(t):
    """GPU/CPU tensor -> float64 numpy values (BF16 decoded exactly)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return decode(bits(t))
    return t.double().numpy()


def oracle_fwd(inp, channels=None):
    """Oracle forward of a ConvInputs (optionally on a subset of channels)."""
    x, w, b, init = inp.x, inp.weight, inp.bias, inp.initial_states
    if channels is not None:
        x = x[:, channels]
        w = w[channels]
        b = b[channels] if b is not None else None
        init = init[:, channels] if init is not None else None
    return oracle.fwd(bits(x), bits(w), bits(b),
                      None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                      bits(init), inp.activation)


def oracle_bwd(inp, channels=None):
    x, w, b, init, g, gf = inp.x, inp.weight, inp.bias, inp.initial_states, inp.g, inp.dfinal_states
    if channels is not None:
        x = x[:, channels]
        g = g[:, channels]
        w = w[channels]
        b = b[channels] if b is not None else None
        init = init[:, channels] if init is not None else None
        gf = gf[:, channels] if gf is not None else None
    return oracle.bwd(bits(x), bits(w), bits(g), bits(b),
                      None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                      bits(init), bits(gf), inp.activation)


def assert_fullconv_close(gpu_bits, ref64, abs_sum, what="full conv out"):
    g = decode(gpu_bits)
    err = np.abs(g - ref64)
    bound = WG_REL * abs_sum + BF16_HALF_ULP_REL * np.abs(ref64) + 1e-30
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst at {i}: "
                             f"gpu={g[i]} ref={ref64[i]} sum|terms|={abs_sum[i]}")
