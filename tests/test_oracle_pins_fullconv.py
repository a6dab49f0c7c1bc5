"""Pins for the oracle of the full-channel dilated causal conv1d (POPCORNBENCH
conv1d page: a Conv1d over all input channels with dilation, left-padded by
P = (K-1)*dilation so that tap k reads input position t + k*dilation - P).

Each check compares the oracle with something other than itself: torch's
conv1d with dilation on the left-padded input (float64), the page's tap
offsets (golden file), impulse responses, the K = 1 case as a plain matrix
product, the depthwise oracle for a diagonal weight, causality, and the
magnitude sums through torch's conv1d of absolute values.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from conftest import golden

RNG = np.random.default_rng(4321)


def _torch_causal(x, w, b, dil):
    K = w.shape[2]
    P = (K - 1) * dil
    xp = F.pad(torch.from_numpy(x), (P, 0))
    return F.conv1d(xp, torch.from_numpy(w), None if b is None else torch.from_numpy(b),
                    dilation=dil).numpy()


@pytest.mark.parametrize("B,Cin,Cout,T,K,dil", [
    (2, 3, 5, 17, 4, 1), (1, 4, 4, 20, 3, 2), (2, 2, 3, 9, 2, 5), (1, 5, 2, 6, 4, 3),
    (1, 3, 3, 1, 4, 2), (2, 1, 1, 12, 1, 1), (1, 6, 4, 33, 5, 4),
])
@pytest.mark.parametrize("with_bias", [False, True])
def test_fullconv_matches_torch_dilated_conv1d(B, Cin, Cout, T, K, dil, with_bias):
    x = RNG.standard_normal((B, Cin, T))
    w = RNG.uniform(-0.5, 0.5, (Cout, Cin, K))
    b = RNG.uniform(-0.1, 0.1, Cout) if with_bias else None
    r = oracle.fullconv_f64(x, w, b, dil)
    np.testing.assert_allclose(r["out"], _torch_causal(x, w, b, dil), rtol=1e-12, atol=1e-13)


def test_fullconv_tap_offsets_from_golden():
    """Tap k reads the input at the page's offset k*dilation - P."""
    for case in golden("tap_order.json")["cases"]:
        K, dil = case["kernel_size"], case["dilation"]
        assert case["padding"] == (K - 1) * dil
        T, t0 = 16, 9
        x = np.zeros((1, 1, T))
        x[0, 0, t0] = 1.0
        for k in range(K):
            w = np.zeros((1, 1, K))
            w[0, 0, k] = 1.0
            out = oracle.fullconv_f64(x, w, None, dil)["out"][0, 0]
            expect = np.zeros(T)
            expect[t0 - case["input_offset_of_tap"][k]] = 1.0
            np.testing.assert_array_equal(out, expect)


def test_fullconv_impulse_response_reads_weight_column():
    Cin, Cout, K, dil, T = 3, 4, 3, 2, 14
    w = RNG.uniform(-0.5, 0.5, (Cout, Cin, K))
    b = RNG.uniform(-0.1, 0.1, Cout)
    for ic in range(Cin):
        x = np.zeros((1, Cin, T))
        x[0, ic, 2] = 1.0
        out = oracle.fullconv_f64(x, w, b, dil)["out"][0]
        expect = np.repeat(b[:, None], T, axis=1)
        for k in range(K):
            expect[:, 2 + (K - 1 - k) * dil] += w[:, ic, k]
        np.testing.assert_allclose(out, expect, rtol=0, atol=1e-15)


def test_fullconv_single_tap_is_a_matrix_product():
    B, Cin, Cout, T = 2, 7, 5, 11
    x = RNG.standard_normal((B, Cin, T))
    w = RNG.uniform(-0.5, 0.5, (Cout, Cin, 1))
    b = RNG.uniform(-0.1, 0.1, Cout)
    out = oracle.fullconv_f64(x, w, b, 3)["out"]
    ref = np.einsum("oi,bit->bot", w[:, :, 0], x) + b[None, :, None]
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-14)


def test_fullconv_diagonal_weight_is_the_depthwise_conv():
    """A diagonal W (W[oc, ic, k] = w[oc, k] when ic == oc) gives the depthwise
    causal conv1d with the identity activation (dilation 1, width four)."""
    B, D, T = 2, 4, 15
    x = RNG.standard_normal((B, D, T))
    w = RNG.uniform(-0.5, 0.5, (D, 4))
    W = np.zeros((D, D, 4))
    for d in range(D):
        W[d, d] = w[d]
    full = oracle.fullconv_f64(x, W, None, 1)["out"]
    dw = oracle.fwd_f64(x, w, None, None, None, None)["out"]
    np.testing.assert_allclose(full, dw, rtol=1e-13, atol=1e-14)


def test_fullconv_causality_bitwise():
    B, Cin, Cout, T, K, dil = 1, 3, 2, 30, 4, 3
    x = RNG.standard_normal((B, Cin, T))
    w = RNG.uniform(-0.5, 0.5, (Cout, Cin, K))
    base = oracle.fullconv_f64(x, w, None, dil)["out"]
    for tp in (0, 5, 17, T - 1):
        x2 = x.copy()
        x2[:, :, tp:] = RNG.standard_normal((B, Cin, T - tp))
        out2 = oracle.fullconv_f64(x2, w, None, dil)["out"]
        assert np.array_equal(out2[:, :, :tp], base[:, :, :tp])
        assert not np.array_equal(out2[:, :, tp:], base[:, :, tp:])


def test_fullconv_abs_sums_match_torch_conv_of_magnitudes():
    B, Cin, Cout, T, K, dil = 2, 4, 3, 19, 3, 2
    x = RNG.standard_normal((B, Cin, T))
    w = RNG.uniform(-0.5, 0.5, (Cout, Cin, K))
    b = RNG.uniform(-0.1, 0.1, Cout)
    r = oracle.fullconv_f64(x, w, b, dil)
    ref = _torch_causal(np.abs(x), np.abs(w), np.abs(b), dil)
    np.testing.assert_allclose(r["abs_sum"], ref, rtol=1e-12, atol=0)


def test_fullconv_bf16_interface_rounds_once():
    B, Cin, Cout, T = 1, 3, 2, 8
    xb = oracle.bf16_encode(RNG.standard_normal((B, Cin, T)))
    wb = oracle.bf16_encode(RNG.uniform(-0.5, 0.5, (Cout, Cin, 2)))
    r = oracle.fullconv(xb, wb, None, 2)
    assert np.array_equal(r["out"], oracle.bf16_encode(r["out64"]))
    ref = _torch_causal(oracle.bf16_decode(xb), oracle.bf16_decode(wb), None, 2)
    np.testing.assert_allclose(r["out64"], ref, rtol=1e-13, atol=1e-14)


def test_fullconv_rejects_bad_kernel_size_or_dilation():
    with pytest.raises(ValueError):
        oracle.fullconv_f64(np.zeros((1, 2, 3)), np.zeros((2, 2, 2)), None, 0)
    with pytest.raises(ValueError):
        oracle.fullconv_f64(np.zeros((1, 2, 3)), np.zeros((2, 3, 2)), None, 1)
