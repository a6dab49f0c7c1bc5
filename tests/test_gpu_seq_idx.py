"""GPU parity of the seq_idx route (cuDNN "Causal Conv1d" page: the seq_idx[B, T]
keyword, mutually exclusive with cu_seqlens).  Reading: tokens of a row with the
same id form one sequence; a tap reads a token of another id as zero; no state.

The CUDA path (through the Python API and autograd) against the oracle on the
same seeded inputs and ids: channel-last rows with four channels a thread and
with one (odd D), time-contiguous rows, ids in runs (lengths 1 upward) and in
no particular order, identity activation, width three, an id tensor with a
token stride, and the deterministic route's bitwise repeatability.
"""

import numpy as np
import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
import oracle
from helpers import assert_bf16_close, assert_wgrad_close, tensor_values
from workloads import bits, make_inputs, seq_ids

pytestmark = pytest.mark.gpu


def run(inp, ids, device, deterministic=None):
    d = inp.to(device)
    x = d.x.detach().requires_grad_(True)
    w = d.weight.detach().requires_grad_(True)
    b = d.bias.detach().requires_grad_(True) if d.bias is not None else None
    out = ccc.causal_conv1d(x, w, b, seq_idx=ids.to(device) if ids.device.type == "cpu" else ids,
                            activation=inp.activation, deterministic=deterministic)
    out.backward(d.g)
    ccc.check_status(device)
    torch.cuda.synchronize()
    return dict(out=out.detach().cpu(), dx=x.grad.cpu(), dw=w.grad.cpu(),
                db=None if b is None else b.grad.cpu(), out_stride=out.stride(), x_stride=x.stride())


def check(inp, ids, res):
    ids_np = ids.cpu().numpy()
    rf = oracle.fwd(bits(inp.x), bits(inp.weight), bits(inp.bias), None, None, inp.activation,
                    seq_idx=ids_np)
    rb = oracle.bwd(bits(inp.x), bits(inp.weight), bits(inp.g), bits(inp.bias), None, None, None,
                    inp.activation, seq_idx=ids_np)
    assert res["out_stride"] == res["x_stride"]
    assert_bf16_close(bits(res["out"]), rf["out"], "out")
    assert_bf16_close(bits(res["dx"]), rb["dx"], "dx")
    bf16_w = inp.weight.dtype == torch.bfloat16
    assert_wgrad_close(tensor_values(res["dw"]), rb["dw64"], rb["dw_abs"], bf16_w, "dweight")
    if inp.bias is not None:
        assert_wgrad_close(tensor_values(res["db"]), rb["db64"], rb["db_abs"], True, "dbias")


CASES = [
    # (B, D, T, channel_last, id layout, options)
    (3, 264, 300, True, dict(kind="runs", max_run=40), {}),
    (2, 264, 300, True, dict(kind="runs", max_run=1), {}),          # every token its own sequence
    (2, 128, 257, True, dict(kind="random", n_ids=2), {}),
    (2, 37, 150, True, dict(kind="runs", max_run=9), {}),           # odd D: one channel a thread
    (1, 512, 1100, True, dict(kind="runs", max_run=300), dict(bias=False, weight_dtype=torch.float32)),
    (2, 64, 90, True, dict(kind="runs", max_run=7), dict(activation=None)),
    (2, 40, 300, False, dict(kind="runs", max_run=50), {}),         # time-contiguous
    (3, 24, 264, False, dict(kind="random", n_ids=3), {}),
    (1, 9, 77, False, dict(kind="runs", max_run=2), dict(bias=False, weight_dtype=torch.float32)),
    (2, 72, 200, True, dict(kind="runs", max_run=20), dict(width=3)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}D{c[1]}T{c[2]}{'cl' if c[3] else 'bdt'}-{c[4]['kind']}")
def test_seq_idx_parity(case, cuda_device):
    B, D, T, cl, idk, opts = case
    seed = 7 * B + D + T
    inp = make_inputs(B, D, T, channel_last=cl, seed=seed, grad=True, **opts)
    ids = seq_ids(B, T, seed, **idk)
    res = run(inp, ids, cuda_device)
    check(inp, ids, res)


def test_seq_idx_strided_ids(cuda_device):
    """An id tensor that is a strided view (token stride 2, batch stride 3T)."""
    B, D, T = 2, 96, 180
    inp = make_inputs(B, D, T, seed=5, grad=True)
    base = seq_ids(B, 3 * T, 5, kind="runs", max_run=30)
    ids_dev = base.to(cuda_device)[:, : 2 * T : 2]
    assert ids_dev.stride() == (3 * T, 2)
    res = run(inp, ids_dev, cuda_device)
    check(inp, ids_dev.cpu().contiguous(), res)


def test_seq_idx_constant_ids_equal_plain_call(cuda_device):
    """One id for every token: the same results as the call without ids --
    out and dx bitwise (every token takes the same operations in the same
    order; only the weight sums' block partition may differ)."""
    B, D, T = 2, 128, 200
    inp = make_inputs(B, D, T, seed=9, grad=True)
    ids = torch.full((B, T), 4, dtype=torch.int32)
    a = run(inp, ids, cuda_device)
    d = inp.to(cuda_device)
    x = d.x.detach().requires_grad_(True)
    out = ccc.causal_conv1d(x, d.weight, d.bias)
    out.backward(d.g)
    assert torch.equal(a["out"], out.detach().cpu()), "out vs plain call"
    assert torch.equal(a["dx"], x.grad.cpu()), "dx vs plain call"


def test_seq_idx_deterministic_repeats_bitwise(cuda_device):
    B, D, T = 2, 256, 600
    inp = make_inputs(B, D, T, seed=11, grad=True, bias=False)
    ids = seq_ids(B, T, 11, kind="runs", max_run=100)
    first = run(inp, ids, cuda_device, deterministic=True)
    for _ in range(4):
        again = run(inp, ids, cuda_device, deterministic=True)
        assert torch.equal(again["dw"], first["dw"])
        assert torch.equal(again["dx"], first["dx"])


def test_seq_idx_dense_state_size_sampled_channels(cuda_device):
    """The dense_state shape (x stored [4, 2048, 1536] channel-last) with ids in
    runs of up to 512 tokens; channels are independent, so whole sampled
    channels are checked element by element against the oracle."""
    B, D, T = 4, 1536, 2048
    inp = make_inputs(B, D, T, seed=2, grad=True)
    ids = seq_ids(B, T, 2, kind="runs", max_run=512)
    res = run(inp, ids, cuda_device)
    chans = [0, 1, 7, 8, 500, 767, 768, 1535]
    ids_np = ids.numpy()
    sub = lambda t: None if t is None else t[:, chans]
    rf = oracle.fwd(bits(sub(inp.x)), bits(inp.weight[chans]), bits(inp.bias[chans]), None, None,
                    "silu", seq_idx=ids_np)
    rb = oracle.bwd(bits(sub(inp.x)), bits(inp.weight[chans]), bits(sub(inp.g)),
                    bits(inp.bias[chans]), None, None, None, "silu", seq_idx=ids_np)
    assert_bf16_close(bits(res["out"][:, chans]), rf["out"], "out (sampled channels)")
    assert_bf16_close(bits(res["dx"][:, chans]), rb["dx"], "dx (sampled channels)")
    assert_wgrad_close(tensor_values(res["dw"][chans]), rb["dw64"], rb["dw_abs"], True, "dweight")
    assert_wgrad_close(tensor_values(res["db"][chans]), rb["db64"], rb["db_abs"], True, "dbias")
