"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check compares the oracle with an independent statement of the same fact:
brute-force dense matrix products, a library routine (torch's grouped conv1d
and autograd in float64), the full-channel formula printed on the
POPCORNBENCH conv1d page instantiated with a diagonal weight, closed forms,
invariants the cuDNN "Causal Conv1d" page fixes (causality, final-state
identity, state hand-off to causal_conv1d_update, packed == per-sequence),
central finite differences in float64, and torch's own BF16 rounding.
"""

import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from conftest import golden

RNG = np.random.default_rng(1234)


def _bf16_bits(a):
    """Round float64 -> BF16 with torch (float64 -> float32 -> bf16; callers pass
    values exactly representable in float32)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(shape, scale=1.0):
    return _bf16_bits(RNG.standard_normal(shape) * scale)


def _silu(p):
    return p / (1.0 + np.exp(-p))


# ---- number format ---------------------------------------------------------------


def test_bf16_encode_matches_torch_rounding_of_float32_values():
    vals = np.concatenate([
        RNG.standard_normal(20000),
        RNG.standard_normal(2000) * 1e-38,       # float32 subnormal / tiny range
        RNG.standard_normal(2000) * 1e30,
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-45, 1e-40]),
    ]).astype(np.float32)
    # exact ties: 1 + odd multiple of 2^-8 sits halfway between two BF16 values
    ties = np.array([1 + k * 2.0 ** -8 for k in range(1, 64, 2)], dtype=np.float32)
    vals = np.concatenate([vals, ties, -ties])
    ours = oracle.bf16_encode(vals.astype(np.float64))
    ref = _bf16_bits(vals)
    assert np.array_equal(ours, ref)


def test_bf16_encode_fixed_points():
    enc = lambda v: int(oracle.bf16_encode(np.array([v]))[0])
    assert enc(1.0) == 0x3F80
    assert enc(1 + 2.0 ** -8) == 0x3F80          # tie -> even
    assert enc(1 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (upwards)
    assert enc(-2.0) == 0xC000
    assert enc(2.0 ** -133) == 0x0001            # smallest subnormal
    assert enc(2.0 ** -134) == 0x0000            # tie with zero -> even (zero)
    assert enc(255.5 * 2.0 ** 120) == 0x7F80     # rounds up to 2^128 -> inf
    assert enc(255.0 * 2.0 ** 120) == 0x7F7F     # largest finite
    assert enc(-0.0) == 0x8000
    # a value that double-rounds wrongly via float32: 1 + 2^-8 + 2^-40
    assert enc(1 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81


def test_bf16_decode_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((bits & 0x7F80) != 0x7F80)
    dec = oracle.bf16_decode(bits[finite])
    assert np.array_equal(oracle.bf16_encode(dec), bits[finite])


# ---- forward ---------------------------------------------------------------------


def _toeplitz_pre(x, w, b, init):
    """Brute force: per channel, the T x (T+3) banded matrix times the extended
    sequence.  x [B,D,T] float64, w [D,4], b [D] or None, init [B,D,3] or None."""
    B, D, T = x.shape
    pre = np.zeros((B, D, T))
    for bb in range(B):
        for d in range(D):
            xe = np.concatenate([init[bb, d] if init is not None else np.zeros(3), x[bb, d]])
            M = np.zeros((T, T + 3))
            for t in range(T):
                for k in range(4):
                    M[t, t + k] = w[d, k]
            pre[bb, d] = M @ xe + (b[d] if b is not None else 0.0)
    return pre


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 9, 16])
@pytest.mark.parametrize("with_init,with_bias", [(False, False), (True, True), (True, False)])
def test_fwd_matches_toeplitz_brute_force(T, with_init, with_bias):
    B, D = 2, 3
    x = RNG.standard_normal((B, D, T))
    w = RNG.uniform(-0.5, 0.5, (D, 4))
    b = RNG.uniform(-0.1, 0.1, D) if with_bias else None
    init = RNG.standard_normal((B, D, 3)) if with_init else None
    ref_pre = _toeplitz_pre(x, w, b, init)
    for act in ("silu", None):
        r = oracle.fwd_f64(x, w, b, None, init, act)
        np.testing.assert_allclose(r["pre"], ref_pre, rtol=1e-13, atol=1e-14)
        ref_out = _silu(ref_pre) if act else ref_pre
        np.testing.assert_allclose(r["out"], ref_out, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("lengths", [[5], [1, 2, 3], [4, 1, 7, 2], [3, 3]])
def test_fwd_matches_torch_grouped_conv1d(lengths):
    """Library pin: a depthwise conv1d is torch's conv1d with groups == channels,
    applied to the extended sequence (initial state as left padding)."""
    D = 4
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    x = RNG.standard_normal((1, D, T))
    w = RNG.uniform(-0.5, 0.5, (D, 4))
    b = RNG.uniform(-0.1, 0.1, D)
    init = RNG.standard_normal((len(lengths), D, 3))
    r = oracle.fwd_f64(x, w, b, cu, init, "silu")
    for n, L in enumerate(lengths):
        xs = torch.from_numpy(x[:, :, cu[n]:cu[n + 1]])
        xe = torch.cat([torch.from_numpy(init[n:n + 1]), xs], dim=2)
        ref = F.silu(F.conv1d(xe, torch.from_numpy(w)[:, None, :], torch.from_numpy(b), groups=D))
        np.testing.assert_allclose(r["out"][:, :, cu[n]:cu[n + 1]], ref.numpy(), rtol=1e-13, atol=1e-14)
        fin_ref = xe[0, :, -3:].numpy()
        np.testing.assert_array_equal(r["final"][n], fin_ref)


def test_fwd_matches_full_channel_formula_with_diagonal_weight():
    """The POPCORNBENCH page's full-channel causal conv: out[b,oc,t] = sum over
    (ic, k) of W[oc,ic,k] * input[b,ic,t + k*dil - P], zero where the position is
    negative.  A diagonal W (W[oc,ic,k] = w[oc,k] if ic == oc) makes it depthwise."""
    spec = golden("tap_order.json")["cases"][0]
    K, dil, P = spec["kernel_size"], spec["dilation"], spec["padding"]
    B, D, T = 2, 3, 7
    x = RNG.standard_normal((B, D, T))
    w = RNG.uniform(-0.5, 0.5, (D, K))
    Wfull = np.zeros((D, D, K))
    for oc in range(D):
        Wfull[oc, oc] = w[oc]
    ref = np.zeros((B, D, T))
    for b, oc, t in itertools.product(range(B), range(D), range(T)):
        s = 0.0
        for ic in range(D):
            for k in range(K):
                pos = t + k * dil - P
                if pos >= 0:
                    s += Wfull[oc, ic, k] * x[b, ic, pos]
        ref[b, oc, t] = s
    r = oracle.fwd_f64(x, w, None, None, None, None)
    np.testing.assert_allclose(r["out"], ref, rtol=1e-13, atol=1e-14)


def test_tap_order_from_golden():
    """Tap k reads the input at offset k - 3 (tap 3 is the current token)."""
    offsets = golden("tap_order.json")["cases"][0]["input_offset_of_tap"]
    D, T = 1, 8
    x = np.zeros((1, D, T))
    x[0, 0, 4] = 1.0  # impulse at t = 4
    for k in range(4):
        w = np.zeros((D, 4))
        w[0, k] = 1.0
        out = oracle.fwd_f64(x, w, None, None, None, None)["out"][0, 0]
        # tap k at output t reads x[t + offset_k]; the impulse shows at t = 4 - offset_k
        expect = np.zeros(T)
        expect[4 - offsets[k]] = 1.0
        np.testing.assert_array_equal(out, expect)


def test_causality_bitwise():
    B, D, T = 2, 5, 24
    x = _rand_bf16((B, D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    init = _rand_bf16((B, D, 3))
    base = oracle.fwd(x, w, b, None, init)["out"]
    for tp in (0, 3, 11, T - 1):
        x2 = x.copy()
        x2[:, :, tp:] = _rand_bf16((B, D, T - tp))
        out2 = oracle.fwd(x2, w, b, None, init)["out"]
        assert np.array_equal(out2[:, :, :tp], base[:, :, :tp])
        assert not np.array_equal(out2[:, :, tp:], base[:, :, tp:])


def test_closed_forms_identity_and_shift_taps():
    B, D, T = 2, 4, 10
    x = _rand_bf16((B, D, T))
    init = _rand_bf16((B, D, 3))
    e3 = np.zeros((D, 4), np.float32)
    e3[:, 3] = 1.0
    r = oracle.fwd(x, e3, None, None, init, None)
    assert np.array_equal(r["out"], x)                       # tap 3 only: out = x
    e0 = np.zeros((D, 4), np.float32)
    e0[:, 0] = 1.0
    r = oracle.fwd(x, e0, None, None, init, None)            # tap 0 only: out[t] = xe[t-3]
    xe = np.concatenate([init, x], axis=2)
    assert np.array_equal(r["out"], xe[:, :, :T])
    # zero weight, bias b, silu: out = silu(b) everywhere (closed form)
    b = np.array([0.5, -1.0, 2.0, 0.0])
    r = oracle.fwd_f64(x.astype(np.float64), np.zeros((D, 4)), b, None, None, "silu")
    for d in range(D):
        np.testing.assert_allclose(r["out"][:, d], b[d] / (1 + math.exp(-b[d])), rtol=1e-15)


@pytest.mark.parametrize("T", [0, 1, 2, 3, 4, 7])
@pytest.mark.parametrize("with_init", [False, True])
def test_final_state_is_last_three_extended_inputs(T, with_init):
    B, D = 2, 3
    x = _rand_bf16((B, D, T))
    init = _rand_bf16((B, D, 3)) if with_init else None
    r = oracle.fwd(x, _rand_bf16((D, 4), 0.3), None, None, init)
    ext = np.concatenate([init if with_init else np.zeros((B, D, 3), np.uint16), x], axis=2)
    assert np.array_equal(r["final"], ext[:, :, -3:])
    assert r["final"].shape == (B, D, golden("shapes.json")["width"] - 1)


@pytest.mark.parametrize("split", [0, 1, 2, 3, 5, 11, 12])
def test_split_with_state_handoff_equals_unsplit(split):
    B, D, T = 2, 4, 12
    x = _rand_bf16((B, D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    init = _rand_bf16((B, D, 3))
    full = oracle.fwd(x, w, b, None, init)
    first = oracle.fwd(np.ascontiguousarray(x[:, :, :split]), w, b, None, init)
    second = oracle.fwd(np.ascontiguousarray(x[:, :, split:]), w, b, None, first["final"])
    assert np.array_equal(np.concatenate([first["out"], second["out"]], axis=2), full["out"])
    assert np.array_equal(second["final"], full["final"])


def test_update_chain_equals_full_forward():
    B, D, T = 3, 5, 20
    x = _rand_bf16((B, D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    init = _rand_bf16((B, D, 3))
    full = oracle.fwd(x, w, b, None, init)
    state = init.copy()
    outs = []
    for t in range(T):
        r = oracle.update(np.ascontiguousarray(x[:, :, t]), state, w, b)
        outs.append(r["out"])
        state = r["state"]
    assert np.array_equal(np.stack(outs, axis=2), full["out"])
    assert np.array_equal(state, full["final"])


def test_update_with_fp32_weight_and_identity():
    B, D = 2, 3
    x = _rand_bf16((B, D))
    st = _rand_bf16((B, D, 3))
    w = RNG.uniform(-0.5, 0.5, (D, 4)).astype(np.float32)
    r = oracle.update_f64(oracle.bf16_decode(x), oracle.bf16_decode(st), w.astype(np.float64),
                          None, None)
    xe = np.concatenate([oracle.bf16_decode(st), oracle.bf16_decode(x)[:, :, None]], axis=2)
    np.testing.assert_allclose(r["out"], (xe * w.astype(np.float64)[None]).sum(-1), rtol=1e-14)
    np.testing.assert_array_equal(r["state"], xe[:, :, 1:])


@pytest.mark.parametrize("lengths", [[1], [1, 1, 1], [2, 5, 1, 3], [4, 4, 4], [7, 1, 2, 9]])
def test_packed_equals_per_sequence_dense(lengths):
    D = 3
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    x = _rand_bf16((1, D, T))
    g = _rand_bf16((1, D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    init = _rand_bf16((len(lengths), D, 3))
    gf = _rand_bf16((len(lengths), D, 3))
    pk = oracle.fwd(x, w, b, cu, init)
    pb = oracle.bwd(x, w, g, b, cu, init, gf)
    dw_sum = np.zeros((D, 4))
    db_sum = np.zeros(D)
    for n in range(len(lengths)):
        sl = slice(cu[n], cu[n + 1])
        xs = np.ascontiguousarray(x[:, :, sl])
        gs = np.ascontiguousarray(g[:, :, sl])
        dn = oracle.fwd(xs, w, b, None, init[n:n + 1])
        assert np.array_equal(pk["out"][:, :, sl], dn["out"])
        assert np.array_equal(pk["final"][n:n + 1], dn["final"])
        bn = oracle.bwd(xs, w, gs, b, None, init[n:n + 1], gf[n:n + 1])
        assert np.array_equal(pb["dx"][:, :, sl], bn["dx"])
        assert np.array_equal(pb["dinit"][n:n + 1], bn["dinit"])
        dw_sum += bn["dw64"]
        db_sum += bn["db64"]
    np.testing.assert_allclose(pb["dw64"], dw_sum, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(pb["db64"], db_sum, rtol=1e-12, atol=1e-12)


def test_cu_seqlens_rules_from_golden():
    for case in golden("cu_seqlens_cases.json")["cases"]:
        ok = oracle.check_cu_seqlens(case["cu_seqlens"], case["total"])
        assert ok == case["valid"], case["name"]
        if not case["valid"]:
            x = np.zeros((1, 2, case["total"]), np.uint16)
            with pytest.raises(ValueError):
                oracle.fwd(x, np.zeros((2, 4), np.uint16), None, case["cu_seqlens"])


# ---- backward --------------------------------------------------------------------


def _loss(r, g, gf):
    L = float((r["out"] * g).sum())
    if gf is not None:
        L += float((r["final"] * gf).sum())
    return L


def _fd_case(B, D, T, act, with_init, with_bias, with_gf, lengths=None, seed=0):
    rng = np.random.default_rng(seed)
    if lengths is not None:
        B, T = 1, sum(lengths)
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        S = len(lengths)
    else:
        cu, S = None, B
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.8, 0.8, (D, 4))
    b = rng.uniform(-0.3, 0.3, D) if with_bias else None
    init = rng.standard_normal((S, D, 3)) if with_init else None
    gf = rng.standard_normal((S, D, 3)) if with_gf else None
    return x, g, w, b, cu, init, gf


def _central_diff(fn, arr, h=1e-6):
    grad = np.zeros_like(arr)
    for idx in np.ndindex(arr.shape):
        keep = arr[idx]
        arr[idx] = keep + h
        lp = fn()
        arr[idx] = keep - h
        lm = fn()
        arr[idx] = keep
        grad[idx] = (lp - lm) / (2 * h)
    return grad


FD_CASES = [
    dict(B=2, D=3, T=1, act="silu", with_init=True, with_bias=True, with_gf=True),
    dict(B=2, D=3, T=2, act="silu", with_init=True, with_bias=False, with_gf=True),
    dict(B=2, D=3, T=5, act="silu", with_init=False, with_bias=True, with_gf=False),
    dict(B=2, D=3, T=9, act="silu", with_init=True, with_bias=True, with_gf=True),
    dict(B=1, D=2, T=9, act=None, with_init=True, with_bias=True, with_gf=True),
    dict(B=1, D=2, T=0, act="silu", with_init=True, with_bias=False, with_gf=False,
         lengths=[1, 4, 2, 1]),
    dict(B=1, D=2, T=0, act="silu", with_init=True, with_bias=True, with_gf=True,
         lengths=[3, 1, 5]),
]


@pytest.mark.parametrize("case", FD_CASES, ids=lambda c: f"T{c['T']}-{c['act']}-{c.get('lengths')}")
def test_bwd_matches_central_finite_differences(case):
    x, g, w, b, cu, init, gf = _fd_case(**case)
    act = case["act"]

    def L():
        return _loss(oracle.fwd_f64(x, w, b, cu, init, act), g, gf)

    r = oracle.bwd_f64(x, w, g, b, cu, init, gf, act)
    tol = dict(rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(r["dx"], _central_diff(L, x), **tol)
    np.testing.assert_allclose(r["dw"], _central_diff(L, w), **tol)
    if b is not None:
        np.testing.assert_allclose(r["db"], _central_diff(L, b), **tol)
    if init is not None:
        np.testing.assert_allclose(r["dinit"], _central_diff(L, init), **tol)


def test_bwd_matches_torch_autograd_float64():
    """Library pin: torch autograd through grouped conv1d + silu on the extended
    sequence, dense with initial state and a final-state gradient."""
    rng = np.random.default_rng(7)
    B, D, T = 3, 4, 11
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.5, 0.5, (D, 4))
    b = rng.uniform(-0.1, 0.1, D)
    init = rng.standard_normal((B, D, 3))
    gf = rng.standard_normal((B, D, 3))
    tx, tw, tb, ti = (torch.tensor(a, requires_grad=True) for a in (x, w, b, init))
    xe = torch.cat([ti, tx], dim=2)
    out = F.silu(F.conv1d(xe, tw[:, None, :], tb, groups=D))
    fin = xe[:, :, -3:]
    L = (out * torch.from_numpy(g)).sum() + (fin * torch.from_numpy(gf)).sum()
    L.backward()
    r = oracle.bwd_f64(x, w, g, b, None, init, gf, "silu")
    np.testing.assert_allclose(r["dx"], tx.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dw"], tw.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["db"], tb.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dinit"], ti.grad.numpy(), rtol=1e-12, atol=1e-13)


def _abs_sums_brute_force(x, w, g, b, lengths, init, act):
    """sum_t |gp[t] * xe[t - S + k]| per (channel, tap) and sum_t |gp[t]| per
    channel, by brute force: gp = dL/dpre from torch autograd of
    act(conv1d(xe)) with L = sum(out * g), one sequence at a time (dense rows,
    or the packed ranges), the absolute terms summed with numpy."""
    B, D, T = x.shape
    W = w.shape[1]
    S = W - 1
    if lengths is None:
        seqs = [(bb, 0, T) for bb in range(B)]
    else:
        starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
        seqs = [(0, int(s0), int(n)) for s0, n in zip(starts, lengths)]
    dw_abs = np.zeros((D, W))
    db_abs = np.zeros(D)
    tw = torch.from_numpy(w)[:, None, :]
    tb = torch.from_numpy(b) if b is not None else None
    for n, (row, start, L) in enumerate(seqs):
        if L == 0:
            continue
        xs = torch.from_numpy(x[row:row + 1, :, start:start + L])
        pad = torch.from_numpy(init[n:n + 1]) if init is not None else torch.zeros(1, D, S,
                                                                                  dtype=torch.float64)
        xe = torch.cat([pad, xs], dim=2)                       # xe[j - S] at index j
        pre = F.conv1d(xe, tw, tb, groups=D).detach().requires_grad_(True)
        out = F.silu(pre) if act == "silu" else pre
        (out * torch.from_numpy(g[row:row + 1, :, start:start + L])).sum().backward()
        gp = pre.grad.numpy()[0]                               # [D, L]
        xen = xe.numpy()[0]                                    # [D, L + S]
        for k in range(W):
            dw_abs[:, k] += np.abs(gp * xen[:, k:k + L]).sum(axis=1)
        db_abs += np.abs(gp).sum(axis=1)
    return dw_abs, db_abs


ABS_SUM_CASES = [
    dict(B=2, D=3, T=17, W=4, act="silu", with_init=True, with_bias=True, lengths=None),
    dict(B=3, D=2, T=9, W=4, act="silu", with_init=False, with_bias=False, lengths=None),
    dict(B=1, D=3, T=17, W=4, act="silu", with_init=True, with_bias=False, lengths=[3, 1, 5, 8]),
    dict(B=2, D=3, T=11, W=4, act=None, with_init=True, with_bias=True, lengths=None),
    dict(B=2, D=3, T=10, W=3, act="silu", with_init=True, with_bias=True, lengths=None),
    dict(B=1, D=2, T=12, W=2, act="silu", with_init=True, with_bias=False, lengths=[1, 6, 5]),
]


@pytest.mark.parametrize("case", ABS_SUM_CASES,
                         ids=lambda c: f"W{c['W']}-{c['act']}-{'packed' if c['lengths'] else 'dense'}")
def test_bwd_abs_sums_match_brute_force(case):
    """The weight/bias-gradient tolerance scale (cuDNN page, determinism
    paragraph: dweight is a sum of FP32 terms; the tolerance is relative to the
    sum of their magnitudes) computed independently of the oracle's loops."""
    rng = np.random.default_rng(900 + case["T"] + 10 * case["W"])
    B, D, T, W = case["B"], case["D"], case["T"], case["W"]
    lengths = case["lengths"]
    S = len(lengths) if lengths else B
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.8, 0.8, (D, W))
    b = rng.uniform(-0.3, 0.3, D) if case["with_bias"] else None
    init = rng.standard_normal((S, D, W - 1)) if case["with_init"] else None
    cu = None if lengths is None else np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    r = oracle.bwd_f64(x, w, g, b, cu, init, None, case["act"])
    dw_abs, db_abs = _abs_sums_brute_force(x, w, g, b, lengths, init, case["act"])
    np.testing.assert_allclose(r["dw_abs"], dw_abs, rtol=1e-12, atol=0)
    np.testing.assert_allclose(r["db_abs"], db_abs, rtol=1e-12, atol=0)
    assert np.all(np.abs(r["dw"]) <= r["dw_abs"] * (1 + 1e-12))
    assert np.all(np.abs(r["db"]) <= r["db_abs"] * (1 + 1e-12))


def test_bwd_bf16_interface_rounds_fp64_results():
    B, D, T = 2, 3, 6
    x = _rand_bf16((B, D, T))
    g = _rand_bf16((B, D, T))
    w32 = RNG.uniform(-0.5, 0.5, (D, 4)).astype(np.float32)
    r = oracle.bwd(x, w32, g, None, None, _rand_bf16((B, D, 3)))
    assert r["dw"].dtype == np.float32
    np.testing.assert_array_equal(r["dw"], r["dw64"].astype(np.float32))
    assert np.array_equal(r["dx"], oracle.bf16_encode(r["dx64"]))
    wb = _rand_bf16((D, 4), 0.3)
    r = oracle.bwd(x, wb, g, _rand_bf16((D,), 0.05))
    assert r["dw"].dtype == np.uint16 and r["db"].dtype == np.uint16


# ---- other filter widths (W = 2, 3; the page's tensors are weight[D, W] and
# states [., D, W - 1]) ---------------------------------------------------------


def _toeplitz_pre_w(x, w, b, init):
    """Brute force for any width: the T x (T + W - 1) banded matrix per channel
    times the extended sequence (initial state as its first W - 1 entries)."""
    B, D, T = x.shape
    W = w.shape[1]
    S = W - 1
    pre = np.zeros((B, D, T))
    for bb in range(B):
        for d in range(D):
            xe = np.concatenate([init[bb, d] if init is not None else np.zeros(S), x[bb, d]])
            M = np.zeros((T, T + S))
            for t in range(T):
                M[t, t:t + W] = w[d]
            pre[bb, d] = M @ xe + (b[d] if b is not None else 0.0)
    return pre


@pytest.mark.parametrize("W", [2, 3])
@pytest.mark.parametrize("T", [1, 2, 5, 9])
def test_fwd_other_widths_match_toeplitz_brute_force(W, T):
    B, D = 2, 3
    x = RNG.standard_normal((B, D, T))
    w = RNG.uniform(-0.5, 0.5, (D, W))
    b = RNG.uniform(-0.1, 0.1, D)
    init = RNG.standard_normal((B, D, W - 1))
    r = oracle.fwd_f64(x, w, b, None, init, "silu")
    ref = _toeplitz_pre_w(x, w, b, init)
    np.testing.assert_allclose(r["pre"], ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["out"], _silu(ref), rtol=1e-13, atol=1e-14)
    xe = np.concatenate([init, x], axis=2)
    np.testing.assert_array_equal(r["final"], xe[:, :, -(W - 1):])


@pytest.mark.parametrize("W", [2, 3, 4])
def test_fwd_widths_match_torch_grouped_conv1d_packed(W):
    lengths = [4, 1, 6]
    D, T = 3, 11
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    x = RNG.standard_normal((1, D, T))
    w = RNG.uniform(-0.5, 0.5, (D, W))
    b = RNG.uniform(-0.1, 0.1, D)
    init = RNG.standard_normal((len(lengths), D, W - 1))
    r = oracle.fwd_f64(x, w, b, cu, init, "silu")
    for n in range(len(lengths)):
        xe = torch.cat([torch.from_numpy(init[n:n + 1]), torch.from_numpy(x[:, :, cu[n]:cu[n + 1]])], dim=2)
        ref = F.silu(F.conv1d(xe, torch.from_numpy(w)[:, None, :], torch.from_numpy(b), groups=D))
        np.testing.assert_allclose(r["out"][:, :, cu[n]:cu[n + 1]], ref.numpy(), rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(r["final"][n], xe[0, :, -(W - 1):].numpy())


@pytest.mark.parametrize("W", [2, 3])
def test_update_chain_equals_forward_other_widths(W):
    B, D, T = 2, 4, 9
    x = _rand_bf16((B, D, T))
    w = _rand_bf16((D, W), 0.3)
    b = _rand_bf16((D,), 0.05)
    init = _rand_bf16((B, D, W - 1))
    full = oracle.fwd(x, w, b, None, init)
    state, outs = init.copy(), []
    for t in range(T):
        r = oracle.update(np.ascontiguousarray(x[:, :, t]), state, w, b)
        outs.append(r["out"])
        state = r["state"]
    assert np.array_equal(np.stack(outs, axis=2), full["out"])
    assert np.array_equal(state, full["final"])


@pytest.mark.parametrize("W", [2, 3])
@pytest.mark.parametrize("case", [dict(B=2, D=2, T=1), dict(B=2, D=2, T=6), dict(B=1, D=2, T=0, lengths=[1, 3, 2])],
                         ids=["T1", "T6", "packed"])
def test_bwd_other_widths_match_central_finite_differences(W, case):
    rng = np.random.default_rng(W * 10 + case["T"])
    lengths = case.get("lengths")
    if lengths is not None:
        B, T = 1, sum(lengths)
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        S = len(lengths)
    else:
        B, T, cu, S = case["B"], case["T"], None, case["B"]
    D = case["D"]
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.8, 0.8, (D, W))
    b = rng.uniform(-0.3, 0.3, D)
    init = rng.standard_normal((S, D, W - 1))
    gf = rng.standard_normal((S, D, W - 1))

    def L():
        return _loss(oracle.fwd_f64(x, w, b, cu, init, "silu"), g, gf)

    r = oracle.bwd_f64(x, w, g, b, cu, init, gf, "silu")
    tol = dict(rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(r["dx"], _central_diff(L, x), **tol)
    np.testing.assert_allclose(r["dw"], _central_diff(L, w), **tol)
    np.testing.assert_allclose(r["db"], _central_diff(L, b), **tol)
    np.testing.assert_allclose(r["dinit"], _central_diff(L, init), **tol)


@pytest.mark.parametrize("W", [2, 3])
def test_bwd_other_widths_match_torch_autograd_float64(W):
    rng = np.random.default_rng(70 + W)
    B, D, T = 2, 3, 8
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.5, 0.5, (D, W))
    b = rng.uniform(-0.1, 0.1, D)
    init = rng.standard_normal((B, D, W - 1))
    gf = rng.standard_normal((B, D, W - 1))
    tx, tw, tb, ti = (torch.tensor(a, requires_grad=True) for a in (x, w, b, init))
    xe = torch.cat([ti, tx], dim=2)
    out = F.silu(F.conv1d(xe, tw[:, None, :], tb, groups=D))
    L = (out * torch.from_numpy(g)).sum() + (xe[:, :, -(W - 1):] * torch.from_numpy(gf)).sum()
    L.backward()
    r = oracle.bwd_f64(x, w, g, b, None, init, gf, "silu")
    for got, ref in ((r["dx"], tx.grad), (r["dw"], tw.grad), (r["db"], tb.grad), (r["dinit"], ti.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_widths_outside_two_to_four_are_rejected():
    with pytest.raises(ValueError):
        oracle.fwd_f64(np.zeros((1, 2, 3)), np.zeros((2, 5)))
    with pytest.raises(ValueError):
        oracle.fwd_f64(np.zeros((1, 2, 3)), np.zeros((2, 1)))


# ---- per-token sequence ids (the cuDNN page's seq_idx[B, T] keyword) ------------
#
# Reading: tokens of a row carrying the same id form one sequence; a tap reads
# another sequence's token as zero.  The pins below do not depend on that
# reading's implementation in the oracle: a masked banded matrix, packed
# cu_seqlens calls and per-run dense calls, finite differences and autograd.


def _masked_band_pre(x, w, b, ids):
    """Brute force: per row and channel, the T x T matrix whose entry (t, j) is
    w[j - t + S] when 0 <= t - j <= S and tokens j and t carry the same id."""
    B, D, T = x.shape
    W = w.shape[1]
    S = W - 1
    pre = np.zeros((B, D, T))
    for bb in range(B):
        M = np.zeros((D, T, T))
        for t in range(T):
            for j in range(max(0, t - S), t + 1):
                if ids[bb, j] == ids[bb, t]:
                    M[:, t, j] = w[:, j - t + S]
        for d in range(D):
            pre[bb, d] = M[d] @ x[bb, d] + (b[d] if b is not None else 0.0)
    return pre


def _runs(lengths, first=0, step=1):
    return np.repeat(first + step * np.arange(len(lengths)), lengths).astype(np.int32)


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("kind", ["runs", "random"])
def test_seq_idx_matches_masked_band_matrix(W, kind):
    rng = np.random.default_rng(40 + W)
    B, D, T = 2, 3, 19
    x = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.5, 0.5, (D, W))
    b = rng.uniform(-0.1, 0.1, D)
    if kind == "runs":
        ids = np.stack([_runs([4, 1, 6, 8]), _runs([1, 1, 17], first=7, step=3)])
    else:  # ids need not form runs: equality alone decides
        ids = rng.integers(0, 3, (B, T)).astype(np.int32)
    ref = _masked_band_pre(x, w, b, ids)
    for act in ("silu", None):
        r = oracle.fwd_f64(x, w, b, None, None, act, seq_idx=ids)
        np.testing.assert_allclose(r["pre"], ref, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(r["out"], _silu(ref) if act else ref, rtol=1e-13, atol=1e-14)
        assert r["final"] is None


@pytest.mark.parametrize("lengths", [[1], [3, 1, 5, 2, 7], [2, 2, 2, 2], [1, 1, 1, 9]])
def test_seq_idx_runs_equal_packed_cu_seqlens(lengths):
    D = 3
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    ids = _runs(lengths, first=-5, step=4)[None]  # any int32 values
    x = _rand_bf16((1, D, T))
    g = _rand_bf16((1, D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    pf = oracle.fwd(x, w, b, cu)
    sf = oracle.fwd(x, w, b, seq_idx=ids)
    assert np.array_equal(sf["out"], pf["out"])
    pb = oracle.bwd(x, w, g, b, cu)
    sb = oracle.bwd(x, w, g, b, seq_idx=ids)
    assert np.array_equal(sb["dx"], pb["dx"])
    np.testing.assert_allclose(sb["dw64"], pb["dw64"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sb["db64"], pb["db64"], rtol=1e-13, atol=1e-13)


def test_seq_idx_rows_equal_per_run_dense_calls():
    D = 4
    rows = [[5, 2, 9], [16], [1, 15]]
    T = 16
    ids = np.stack([_runs(r, first=10 * i) for i, r in enumerate(rows)])
    x = _rand_bf16((len(rows), D, T))
    g = _rand_bf16((len(rows), D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    sf = oracle.fwd(x, w, b, seq_idx=ids)
    sb = oracle.bwd(x, w, g, b, seq_idx=ids)
    dw = np.zeros((D, 4))
    for bb, lens in enumerate(rows):
        s0 = 0
        for L in lens:
            sl = slice(s0, s0 + L)
            xs = np.ascontiguousarray(x[bb:bb + 1, :, sl])
            gs = np.ascontiguousarray(g[bb:bb + 1, :, sl])
            assert np.array_equal(sf["out"][bb:bb + 1, :, sl], oracle.fwd(xs, w, b)["out"])
            rb = oracle.bwd(xs, w, gs, b)
            assert np.array_equal(sb["dx"][bb:bb + 1, :, sl], rb["dx"])
            dw += rb["dw64"]
            s0 += L
    np.testing.assert_allclose(sb["dw64"], dw, rtol=1e-12, atol=1e-12)


def test_seq_idx_constant_equals_dense():
    B, D, T = 2, 3, 12
    x = _rand_bf16((B, D, T))
    g = _rand_bf16((B, D, T))
    w = _rand_bf16((D, 4), 0.3)
    b = _rand_bf16((D,), 0.05)
    ids = np.full((B, T), 3, np.int32)
    assert np.array_equal(oracle.fwd(x, w, b, seq_idx=ids)["out"], oracle.fwd(x, w, b)["out"])
    sb, db = oracle.bwd(x, w, g, b, seq_idx=ids), oracle.bwd(x, w, g, b)
    assert np.array_equal(sb["dx"], db["dx"])
    assert np.array_equal(sb["dw64"], db["dw64"])


@pytest.mark.parametrize("kind", ["runs", "random"])
def test_seq_idx_bwd_matches_central_finite_differences(kind):
    rng = np.random.default_rng(55)
    B, D, T = 2, 2, 11
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.8, 0.8, (D, 4))
    b = rng.uniform(-0.3, 0.3, D)
    ids = (np.stack([_runs([3, 1, 7]), _runs([6, 5])]) if kind == "runs"
           else rng.integers(0, 2, (B, T)).astype(np.int32))

    def L():
        return float((oracle.fwd_f64(x, w, b, None, None, "silu", seq_idx=ids)["out"] * g).sum())

    r = oracle.bwd_f64(x, w, g, b, None, None, None, "silu", seq_idx=ids)
    tol = dict(rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(r["dx"], _central_diff(L, x), **tol)
    np.testing.assert_allclose(r["dw"], _central_diff(L, w), **tol)
    np.testing.assert_allclose(r["db"], _central_diff(L, b), **tol)


def test_seq_idx_bwd_matches_torch_autograd_float64():
    """Autograd through the taps written with a per-tap id mask."""
    rng = np.random.default_rng(77)
    B, D, T, W = 2, 3, 14, 4
    S = W - 1
    x = rng.standard_normal((B, D, T))
    g = rng.standard_normal((B, D, T))
    w = rng.uniform(-0.5, 0.5, (D, W))
    b = rng.uniform(-0.1, 0.1, D)
    ids = np.stack([_runs([2, 5, 7]), rng.integers(0, 3, T).astype(np.int32)])
    tx, tw, tb = (torch.tensor(a, requires_grad=True) for a in (x, w, b))
    pre = tb[None, :, None].expand(B, D, T).clone()
    for k in range(W):
        sh = S - k  # tap k reads position t - sh
        xs = F.pad(tx, (sh, 0))[:, :, :T]
        m = np.zeros((B, T))
        for bb in range(B):
            for t in range(sh, T):
                m[bb, t] = ids[bb, t - sh] == ids[bb, t]
        pre = pre + tw[None, :, k:k + 1] * xs * torch.from_numpy(m)[:, None, :]
    (F.silu(pre) * torch.from_numpy(g)).sum().backward()
    r = oracle.bwd_f64(x, w, g, b, None, None, None, "silu", seq_idx=ids)
    np.testing.assert_allclose(r["dx"], tx.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["dw"], tw.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["db"], tb.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_seq_idx_declines_packed_and_states():
    """The page makes seq_idx and cu_seqlens mutually exclusive; no state is
    defined with seq_idx."""
    x = np.zeros((1, 2, 4))
    w = np.zeros((2, 4))
    ids = np.zeros((1, 4), np.int32)
    with pytest.raises(ValueError):
        oracle.fwd_f64(x, w, None, np.array([0, 4], np.int32), None, "silu", seq_idx=ids)
    with pytest.raises(ValueError):
        oracle.fwd_f64(x, w, None, None, np.zeros((1, 2, 3)), "silu", seq_idx=ids)
    with pytest.raises(ValueError):
        oracle.bwd_f64(x, w, x, None, None, None, np.zeros((1, 2, 3)), "silu", seq_idx=ids)
    with pytest.raises(ValueError):
        oracle.fwd_f64(x, w, None, None, None, "silu", seq_idx=np.zeros((1, 3), np.int32))
