"""GPU parity: the CUDA path against the CPU oracle on identical seeded inputs.

Sizes are small enough for the oracle to finish in seconds but span several
thread blocks along channels and tokens, with ragged tails.  Bars (see
helpers.py): final states and update state bit-exact; BF16 results within
1e-2 + 1.6e-2 |ref| of the oracle rounded to BF16; dweight/dbias within
1e-3 sum|terms| (+ one BF16 rounding for BF16 outputs).
"""

import numpy as np
import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
import oracle
from helpers import (assert_bf16_close, assert_bits_equal, assert_wgrad_close, oracle_bwd,
                     oracle_fwd, tensor_values)
from workloads import bits, make_inputs

pytestmark = pytest.mark.gpu


def gpu_run(inp, device, backward=True, deterministic=None):
    """Forward (+ backward through autograd) on the GPU; returns CPU tensors."""
    d = inp.to(device)
    x = d.x.detach().requires_grad_(backward)
    w = d.weight.detach().requires_grad_(backward)
    b = d.bias.detach().requires_grad_(backward) if d.bias is not None else None
    init = d.initial_states.detach().requires_grad_(backward) if d.initial_states is not None else None
    out, fin = ccc.causal_conv1d(x, w, b, cu_seqlens=d.cu_seqlens, initial_states=init,
                                 return_final_states=True, activation=d.activation,
                                 deterministic=deterministic)
    res = dict(out=out.detach().cpu(), final=fin.detach().cpu(), out_stride=out.stride(),
               x_stride=x.stride())
    if backward:
        grads = [d.g]
        outs = [out]
        if d.dfinal_states is not None:
            outs.append(fin)
            grads.append(d.dfinal_states)
        torch.autograd.backward(outs, grads)
        res.update(dx=x.grad.cpu(), dw=w.grad.cpu(), db=None if b is None else b.grad.cpu(),
                   dinit=None if init is None else init.grad.cpu(), dx_stride=x.grad.stride())
    ccc.check_status(device)
    torch.cuda.synchronize()
    return res


def check_fwd(inp, res):
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(res["out"]), ref["out"], "out")
    assert_bits_equal(bits(res["final"]), ref["final"], "final_states")
    assert res["out_stride"] == res["x_stride"]


def check_bwd(inp, res):
    ref = oracle_bwd(inp)
    assert_bf16_close(bits(res["dx"]), ref["dx"], "dx")
    assert res["dx_stride"] == res["x_stride"]
    bf16_w = inp.weight.dtype == torch.bfloat16
    assert res["dw"].dtype == inp.weight.dtype
    assert_wgrad_close(tensor_values(res["dw"]), ref["dw64"], ref["dw_abs"], bf16_w, "dweight")
    if inp.bias is not None:
        assert_wgrad_close(tensor_values(res["db"]), ref["db64"], ref["db_abs"], True, "dbias")
    if inp.initial_states is not None:
        assert_bf16_close(bits(res["dinit"]), ref["dinit"], "dinitial_states")


DENSE_CASES = [
    # (B, D, T, channel_last, options)
    # eight channels a thread in blocks two warps wide, the last block column
    # one channel group wide (D = 4104 = 64 * 64 + 8)
    (1, 4104, 12000, True, dict(initial_states=True, grad=True)),
    # dense plans cut each sequence into its own segments: many short
    # sequences (one segment each, shorter than a planned segment), and
    # sequences whose last segment is ragged, with states in and out
    (48, 512, 7, True, dict(initial_states=True, grad=True, dfinal_states=True)),
    (64, 256, 1, True, dict(initial_states=True, grad=True, dfinal_states=True)),
    (33, 136, 2, True, dict(initial_states=True, grad=True, dfinal_states=True)),
    (5, 1024, 997, True, dict(initial_states=True, grad=True, dfinal_states=True)),
    (3, 264, 300, True, dict(initial_states=True, grad=True)),
    (2, 264, 300, True, dict(initial_states=True, grad=True, dfinal_states=True)),
    (2, 64, 37, True, dict(grad=True)),
    (1, 1024, 129, True, dict(initial_states=True, grad=True, bias=False, weight_dtype=torch.float32)),
    (2, 100, 77, True, dict(initial_states=True, grad=True, dfinal_states=True)),      # D % 8 != 0
    (2, 8, 50, True, dict(initial_states=True, grad=True, activation=None)),
    (3, 1, 40, True, dict(initial_states=True, grad=True)),
    (2, 40, 300, False, dict(initial_states=True, grad=True, dfinal_states=True)),     # [B, D, T]
    (2, 64, 128, False, dict(grad=True)),
    (1, 33, 7, False, dict(initial_states=True, grad=True, bias=False, weight_dtype=torch.float32)),
    # time-contiguous rows of a multiple of 8 tokens: 8 tokens a lane, warp steps of 256;
    # an even D takes two channel rows a warp (the last block ragged for 3 x 10)
    (3, 24, 264, False, dict(initial_states=True, grad=True, dfinal_states=True)),
    (2, 16, 512, False, dict(initial_states=True, grad=True)),
    (1, 8, 2056, False, dict(grad=True, activation=None)),
    (3, 10, 520, False, dict(initial_states=True, grad=True, dfinal_states=True)),
    # an odd D: one channel row a warp
    (2, 25, 264, False, dict(initial_states=True, grad=True, dfinal_states=True)),
    (1, 7, 512, False, dict(initial_states=True, grad=True, bias=False, weight_dtype=torch.float32)),
    # rows of 4096 tokens or more: the backward takes two channel rows a warp for an even D
    (2, 6, 4096, False, dict(initial_states=True, grad=True, dfinal_states=True)),
    (1, 10, 4104, False, dict(grad=True, bias=False, weight_dtype=torch.float32)),
    (1, 4, 4096, False, dict(initial_states=True, grad=True, activation=None)),
    (1, 5, 4096, False, dict(initial_states=True, grad=True)),
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: f"B{c[0]}D{c[1]}T{c[2]}{'cl' if c[3] else 'bdt'}")
def test_dense_parity(case, cuda_device):
    B, D, T, cl, opts = case
    inp = make_inputs(B, D, T, channel_last=cl, seed=B * 1000 + D + T, **opts)
    res = gpu_run(inp, cuda_device)
    check_fwd(inp, res)
    check_bwd(inp, res)


@pytest.mark.parametrize("T", [0, 1, 2, 3, 4, 5, 6, 7, 8, 9])
@pytest.mark.parametrize("cl", [True, False])
def test_short_sequences(T, cl, cuda_device):
    inp = make_inputs(2, 16, T, channel_last=cl, seed=T, initial_states=True, grad=True,
                      dfinal_states=True)
    res = gpu_run(inp, cuda_device)
    check_fwd(inp, res)
    check_bwd(inp, res)


PACKED = [
    [1],
    [2],
    [1, 1, 1, 2],
    [5, 1, 2, 300, 7],
    [3, 3, 3, 3, 3, 3],
    [129, 1, 64, 2, 255],
]


@pytest.mark.parametrize("lengths", PACKED, ids=lambda l: "-".join(map(str, l)))
@pytest.mark.parametrize("cl", [True, False])
@pytest.mark.parametrize("deterministic", [False, True])
def test_packed_parity(lengths, cl, deterministic, cuda_device):
    T = sum(lengths)
    inp = make_inputs(1, 72, T, channel_last=cl, seed=len(lengths) + T, lengths=lengths,
                      initial_states=True, grad=True, dfinal_states=True, bias=not deterministic,
                      weight_dtype=torch.float32 if deterministic else torch.bfloat16)
    res = gpu_run(inp, cuda_device, deterministic=deterministic)
    check_fwd(inp, res)
    check_bwd(inp, res)


def test_packed_random_lengths(cuda_device):
    rng = np.random.default_rng(5)
    lengths = rng.integers(1, 200, size=16).tolist()
    T = int(sum(lengths))
    inp = make_inputs(1, 256, T, seed=11, lengths=lengths, initial_states=True, grad=True,
                      bias=False, weight_dtype=torch.float32)
    res = gpu_run(inp, cuda_device, deterministic=True)
    check_fwd(inp, res)
    check_bwd(inp, res)


def test_packed_without_state(cuda_device):
    lengths = [4, 9, 1, 30]
    inp = make_inputs(1, 24, sum(lengths), seed=3, lengths=lengths, grad=True)
    res = gpu_run(inp, cuda_device)
    check_fwd(inp, res)
    check_bwd(inp, res)


def test_time_contiguous_unaligned_rows_take_the_scalar_path(cuda_device):
    """A [B, D, T] view starting one element into its storage: rows are not
    16-byte aligned, so the per-token kernel runs; results match the oracle."""
    B, D, T = 2, 16, 64
    inp = make_inputs(B, D, T, channel_last=False, seed=77, initial_states=True, grad=True)
    big = torch.zeros(B * D * T + 8, dtype=torch.bfloat16)
    big[1:1 + B * D * T] = inp.x.reshape(-1)
    x_un = big[1:1 + B * D * T].view(B, D, T)
    d = inp.to(cuda_device)
    xg = big.to(cuda_device)[1:1 + B * D * T].view(B, D, T).detach().requires_grad_(True)
    assert xg.data_ptr() % 16 != 0
    out, fin = ccc.causal_conv1d(xg, d.weight, d.bias, initial_states=d.initial_states,
                                 return_final_states=True)
    out.backward(d.g)
    ccc.check_status(cuda_device)
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(out.detach().cpu()), ref["out"], "out")
    assert_bits_equal(bits(fin.cpu()), ref["final"], "final")
    assert_bf16_close(bits(xg.grad.cpu()), oracle_bwd(inp)["dx"], "dx")
    assert torch.equal(x_un, inp.x)


def test_unaligned_base_pointer_uses_scalar_path(cuda_device):
    """x and grad_out start one element past a 16-byte boundary."""
    B, D, T = 2, 64, 50
    inp = make_inputs(B, D, T, seed=9, initial_states=True, grad=True)
    d = inp.to(cuda_device)
    buf = torch.empty(B * T * D + 1, dtype=torch.bfloat16, device=cuda_device)
    xs = buf[1:].view(B, T, D)
    xs.copy_(d.x.transpose(1, 2))
    x = xs.transpose(1, 2)
    gbuf = torch.empty(B * T * D + 1, dtype=torch.bfloat16, device=cuda_device)
    gs = gbuf[1:].view(B, T, D)
    gs.copy_(d.g.transpose(1, 2))
    x.requires_grad_(True)
    out, fin = ccc.causal_conv1d(x, d.weight, d.bias, initial_states=d.initial_states,
                                 return_final_states=True)
    out.backward(gs.transpose(1, 2))
    ccc.check_status(cuda_device)
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(out.detach().cpu()), ref["out"], "out")
    assert_bits_equal(bits(fin.cpu()), ref["final"], "final")
    rb = oracle_bwd(inp)
    assert_bf16_close(bits(x.grad.cpu()), rb["dx"], "dx")


def test_forward_only_variants(cuda_device):
    """No final state requested; identity activation; FP32 weight."""
    inp = make_inputs(2, 128, 64, seed=21, bias=False, weight_dtype=torch.float32, activation=None)
    d = inp.to(cuda_device)
    out = ccc.causal_conv1d(d.x, d.weight, None, activation=None)
    ccc.check_status(cuda_device)
    assert_bf16_close(bits(out.cpu()), oracle_fwd(inp)["out"], "out")


def test_final_states_out_argument(cuda_device):
    inp = make_inputs(2, 32, 20, seed=4, initial_states=True)
    d = inp.to(cuda_device)
    buf = torch.full((2, 32, 3), 7.0, dtype=torch.bfloat16, device=cuda_device)
    out, fin = ccc.causal_conv1d(d.x, d.weight, d.bias, initial_states=d.initial_states,
                                 final_states_out=buf)
    assert fin.data_ptr() == buf.data_ptr()
    assert_bits_equal(bits(buf.cpu()), oracle_fwd(inp)["final"], "final_states_out")
    with pytest.raises(ValueError):  # aliasing the initial states is rejected
        ccc.causal_conv1d(d.x, d.weight, d.bias, initial_states=d.initial_states,
                          final_states_out=d.initial_states)


def test_guard_regions_untouched(cuda_device):
    """Outputs sit inside larger buffers filled with a canary; nothing outside
    the outputs may change (stand-in for a memory checker)."""
    from depthwise_causal_conv1d_channel_gb300 import _abi

    B, D, T = 2, 72, 45
    inp = make_inputs(B, D, T, seed=8, initial_states=True, grad=True, dfinal_states=True)
    d = inp.to(cuda_device)
    G = 4096
    canary = -12345

    def guarded(shape, strides_like=None):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * G,), canary, dtype=torch.int16, device=cuda_device)
        core = buf[G:G + n].view(torch.bfloat16)
        if strides_like is not None:  # channel-last [B, T, D] storage
            t = core.view(shape[0], shape[2], shape[1]).transpose(1, 2)
        else:
            t = core.view(*shape)
        return buf, t

    ob, out = guarded((B, D, T), True)
    fb, fin = guarded((B, D, 3))
    assert _abi.ccc_conv1d_fwd(d.x, d.weight, d.bias, None, d.initial_states, out, fin, 1,
                               None, torch.cuda.current_stream()) == 0
    xb, dx = guarded((B, D, T), True)
    ib, dinit = guarded((B, D, 3))
    dw = torch.empty_like(d.weight)
    db = torch.empty_like(d.bias)
    ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(d.x, False), dtype=torch.uint8,
                     device=cuda_device)
    assert _abi.ccc_conv1d_bwd(d.x, d.weight, d.bias, None, d.initial_states, d.g,
                               d.dfinal_states, dx, dw, db, dinit, 1, False, ws, None,
                               torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    for buf in (ob, fb, xb, ib):
        assert bool((buf[:G] == canary).all()) and bool((buf[-G:] == canary).all())
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(out.cpu()), ref["out"], "out")
    rb = oracle_bwd(inp)
    assert_bf16_close(bits(dx.cpu()), rb["dx"], "dx")
    assert_bf16_close(bits(dinit.cpu()), rb["dinit"], "dinit")


def test_deterministic_backward_bitwise_repeatable(cuda_device):
    lengths = [300, 1, 47, 1000, 5]
    inp = make_inputs(1, 512, sum(lengths), seed=13, lengths=lengths, initial_states=True,
                      grad=True, bias=False, weight_dtype=torch.float32)
    first = None
    for _ in range(10):
        res = gpu_run(inp, cuda_device, deterministic=True)
        if first is None:
            first = res
            check_bwd(inp, res)
        else:
            assert torch.equal(res["dw"], first["dw"])
            assert torch.equal(res["dx"].view(torch.int16), first["dx"].view(torch.int16))


def test_default_route_with_bias_is_bitwise_repeatable(cuda_device):
    """The default (non-deterministic flag) route also sums fixed per-block
    partials in a fixed order: dweight and dbias repeat bitwise."""
    inp = make_inputs(3, 520, 700, seed=29, initial_states=True, grad=True)
    first = None
    for _ in range(5):
        res = gpu_run(inp, cuda_device, deterministic=False)
        if first is None:
            first = res
            check_bwd(inp, res)
        else:
            assert torch.equal(res["dw"], first["dw"])
            assert torch.equal(res["db"], first["db"])


def test_deterministic_with_bias_raises(cuda_device):
    inp = make_inputs(1, 16, 8, seed=1, grad=True)
    with pytest.raises(RuntimeError):
        gpu_run(inp, cuda_device, deterministic=True)


def test_use_deterministic_algorithms_flag(cuda_device):
    inp = make_inputs(1, 16, 8, seed=1, grad=True)
    prev = torch.are_deterministic_algorithms_enabled()
    prev_warn = torch.is_deterministic_algorithms_warn_only_enabled()
    try:
        torch.use_deterministic_algorithms(True)
        with pytest.raises(RuntimeError):
            gpu_run(inp, cuda_device)
        torch.use_deterministic_algorithms(True, warn_only=True)
        with pytest.warns(UserWarning):
            res = gpu_run(inp, cuda_device)
        check_bwd(inp, res)
        nb = make_inputs(1, 16, 8, seed=1, grad=True, bias=False)
        torch.use_deterministic_algorithms(True)
        check_bwd(nb, gpu_run(nb, cuda_device))
    finally:
        torch.use_deterministic_algorithms(prev, warn_only=prev_warn)


def test_long_packed_many_short_sequences(cuda_device):
    """Enough tokens per thread that the backward takes its 8-channel path, with
    thousands of sequence boundaries (lengths 1..6), initial states and a
    final-state gradient; a sample of whole channels against the oracle."""
    rng = np.random.default_rng(21)
    lengths = rng.integers(1, 7, size=220_000).tolist()
    T = int(sum(lengths))
    inp = make_inputs(1, 64, T, seed=22, lengths=lengths, initial_states=True, grad=True,
                      dfinal_states=True, bias=False, weight_dtype=torch.float32)
    res = gpu_run(inp, cuda_device, deterministic=True)
    ch = [0, 5, 31, 32, 63]
    idx = torch.tensor(ch)
    rf = oracle_fwd(inp, ch)
    rb = oracle_bwd(inp, ch)
    assert_bf16_close(bits(res["out"][:, idx]), rf["out"], "out")
    assert_bits_equal(bits(res["final"][:, idx]), rf["final"], "final")
    assert_bf16_close(bits(res["dx"][:, idx]), rb["dx"], "dx")
    assert_bf16_close(bits(res["dinit"][:, idx]), rb["dinit"], "dinit")
    assert_wgrad_close(tensor_values(res["dw"][idx]), rb["dw64"], rb["dw_abs"], False, "dweight")


@pytest.mark.parametrize("wdtype", [torch.bfloat16, torch.float32])
def test_strided_weight_and_bias(wdtype, cuda_device):
    """Weight stored transposed ([4, D] memory seen as [D, 4]) and a strided bias:
    the kernels stage them through shared memory instead of vector loads."""
    B, D, T = 2, 136, 90
    inp = make_inputs(B, D, T, seed=41, initial_states=True, grad=True, weight_dtype=wdtype,
                      bias=wdtype == torch.bfloat16)
    d = inp.to(cuda_device)
    w_t = d.weight.t().contiguous().t()                          # strides (1, D)
    assert w_t.stride() == (1, D)
    b_s = None
    if d.bias is not None:
        b_s = torch.zeros(2 * D, dtype=d.bias.dtype, device=cuda_device)[::2]
        b_s.copy_(d.bias)
    x = d.x.detach().requires_grad_(True)
    w = w_t.detach().requires_grad_(True)
    out, fin = ccc.causal_conv1d(x, w, b_s, initial_states=d.initial_states,
                                 return_final_states=True)
    out.backward(d.g)
    ccc.check_status(cuda_device)
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(out.detach().cpu()), ref["out"], "out")
    assert_bits_equal(bits(fin.cpu()), ref["final"], "final")
    rb = oracle_bwd(inp)
    assert_bf16_close(bits(x.grad.cpu()), rb["dx"], "dx")
    assert_wgrad_close(tensor_values(w.grad), rb["dw64"], rb["dw_abs"], wdtype == torch.bfloat16,
                       "dweight")
    st = torch.empty(B, D, 3, dtype=torch.bfloat16, device=cuda_device).copy_(d.initial_states)
    xt = d.x[:, :, 0].contiguous()
    u = ccc.causal_conv1d_update(xt, st, w_t, b_s)
    ru = oracle.update(bits(xt), bits(inp.initial_states), bits(inp.weight), bits(inp.bias))
    assert_bf16_close(bits(u.cpu()), ru["out"], "update out")
