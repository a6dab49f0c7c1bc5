"""The five benchmark workloads at full size, in the launch configuration the
benchmark times.  Channels are independent, so the oracle checks a seeded
sample of whole channels (every token, every sequence) -- exact element-wise
parity on those -- plus properties that hold at any size: final states equal
the last three extended inputs bitwise, the update chain's state equals the
last three tokens, and the deterministic weight gradient is bitwise stable.
"""

import numpy as np
import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
import oracle
import workloads
from helpers import (assert_bf16_close, assert_bits_equal, assert_wgrad_close, oracle_bwd,
                     oracle_fwd, tensor_values)
from workloads import bits

pytestmark = pytest.mark.gpu


def sample_channels(D, n, seed):
    rng = np.random.default_rng(seed)
    ch = set(rng.choice(D, size=min(n, D), replace=False).tolist())
    ch.update({0, D - 1})  # first and last channel always
    return sorted(ch)


def run_fwd_bwd(inp, device, deterministic):
    d = inp.to(device)
    x = d.x.detach().requires_grad_(True)
    w = d.weight.detach().requires_grad_(True)
    b = d.bias.detach().requires_grad_(True) if d.bias is not None else None
    init = d.initial_states.detach().requires_grad_(True)
    out, fin = ccc.causal_conv1d(x, w, b, cu_seqlens=d.cu_seqlens, initial_states=init,
                                 return_final_states=True, deterministic=deterministic)
    out.backward(d.g)
    ccc.check_status(device)
    torch.cuda.synchronize()
    return dict(out=out.detach(), final=fin.detach(), dx=x.grad, dw=w.grad,
                db=None if b is None else b.grad, dinit=init.grad)


def check_sampled(inp, res, channels):
    idx = torch.tensor(channels)
    rf = oracle_fwd(inp, channels)
    rb = oracle_bwd(inp, channels)
    out = res["out"][:, idx.to(res["out"].device)].cpu()
    assert_bf16_close(bits(out), rf["out"], "out")
    assert_bits_equal(bits(res["final"][:, idx.to(res["final"].device)].cpu()), rf["final"], "final")
    assert_bf16_close(bits(res["dx"][:, idx.to(res["dx"].device)].cpu()), rb["dx"], "dx")
    assert_bf16_close(bits(res["dinit"][:, idx.to(res["dinit"].device)].cpu()), rb["dinit"], "dinit")
    bf16_w = inp.weight.dtype == torch.bfloat16
    assert_wgrad_close(tensor_values(res["dw"][idx.to(res["dw"].device)]), rb["dw64"], rb["dw_abs"],
                       bf16_w, "dweight")
    if res["db"] is not None:
        assert_wgrad_close(tensor_values(res["db"][idx.to(res["db"].device)]), rb["db64"],
                           rb["db_abs"], True, "dbias")


def check_final_states_property(inp, res):
    """final[n] == xe[len-3 .. len-1] bitwise for every sequence and channel."""
    x = inp.x  # CPU [B, D, T] view
    fin = bits(res["final"].cpu())
    init = bits(inp.initial_states)
    if inp.cu_seqlens is None:
        B, D, T = x.shape
        tail = bits(x[:, :, max(0, T - 3):])
        ext = np.concatenate([init, tail], axis=2)[:, :, -3:]
        assert_bits_equal(fin, ext, "final_states")
    else:
        cu = inp.cu_seqlens.tolist()
        for n in range(len(cu) - 1):
            tail = bits(x[0, :, max(cu[n], cu[n + 1] - 3):cu[n + 1]])
            ext = np.concatenate([init[n], tail], axis=1)[:, -3:]
            assert_bits_equal(fin[n], ext, f"final_states[{n}]")


def test_dense_small_forward(cuda_device):
    """x [2, 64, 128] contiguous, BF16 weight and bias, no state: every element."""
    inp = workloads.dense_small()
    d = inp.to(cuda_device)
    out = ccc.causal_conv1d(d.x, d.weight, d.bias, activation="silu")
    ccc.check_status(cuda_device)
    assert out.stride() == d.x.stride()
    assert_bf16_close(bits(out.cpu()), oracle_fwd(inp)["out"], "out")


def test_dense_state_fwd_bwd(cuda_device):
    """x stored [4, 2048, 1536] channel-last, initial/final state, default (non-deterministic flag) dW."""
    inp = workloads.dense_state()
    res = run_fwd_bwd(inp, cuda_device, deterministic=False)
    check_sampled(inp, res, sample_channels(1536, 48, 1))
    check_final_states_property(inp, res)
    # the forward output at every element, too (the oracle takes a few seconds)
    assert_bf16_close(bits(res["out"].cpu()), oracle_fwd(inp)["out"], "out (all)")


def test_packed_varlen_deterministic(cuda_device):
    """16 sequences of U[1, 4096] tokens, D = 2048, FP32 weight, no bias,
    deterministic dW; 10 runs bitwise identical."""
    inp = workloads.packed_varlen()
    assert inp.cu_seqlens[-1].item() == inp.x.shape[2]
    res = run_fwd_bwd(inp, cuda_device, deterministic=True)
    check_sampled(inp, res, sample_channels(2048, 24, 2))
    check_final_states_property(inp, res)
    dw0 = res["dw"].clone()
    for _ in range(9):
        r = run_fwd_bwd(inp, cuda_device, deterministic=True)
        assert torch.equal(r["dw"], dw0)


@pytest.mark.parametrize("bias", [True, False], ids=["bias-default", "nobias-deterministic"])
def test_dense_large(bias, cuda_device):
    """x stored [8, 8192, 5120] channel-last; with bias (default route) or
    bias-free deterministic."""
    inp = workloads.dense_large(bias=bias)
    res = run_fwd_bwd(inp, cuda_device, deterministic=not bias)
    check_sampled(inp, res, sample_channels(5120, 12, 3 + bias))
    check_final_states_property(inp, res)
    if not bias:
        dw0 = res["dw"].clone()
        for _ in range(2):
            assert torch.equal(run_fwd_bwd(inp, cuda_device, True)["dw"], dw0)
    del res
    torch.cuda.empty_cache()


def test_decode_update_chain(cuda_device):
    """state [256, 4096, 3], 1000 chained single-token updates; sampled channels
    match the oracle's full-sequence forward; the whole state ends bitwise equal
    to the last three tokens; the GPU chain equals the GPU forward bitwise."""
    wl = workloads.decode_update()
    steps, B, D = wl.x_seq.shape
    x_seq = wl.x_seq.to(cuda_device)
    state = wl.conv_state.to(cuda_device)
    w = wl.weight.to(cuda_device)
    b = wl.bias.to(cuda_device)
    outs = torch.empty(steps, B, D, dtype=torch.bfloat16, device=cuda_device)
    for s in range(steps):
        ccc.causal_conv1d_update(x_seq[s], state, w, b, out=outs[s])
    torch.cuda.synchronize()
    # property at full size: state == last three tokens
    assert torch.equal(state.view(torch.int16),
                       x_seq[-3:].permute(1, 2, 0).contiguous().view(torch.int16))
    # GPU forward over the same sequence ([B, D, T] view of [T, B, D] storage)
    fwd_out = ccc.causal_conv1d(x_seq.permute(1, 2, 0), w, b,
                                initial_states=wl.conv_state.to(cuda_device))
    assert torch.equal(fwd_out.view(torch.int16), outs.permute(1, 2, 0).view(torch.int16))
    # sampled parity with the oracle
    rows = [0, 17, 255]
    chans = sample_channels(D, 16, 5)
    xs = wl.x_seq[:, rows][:, :, chans].permute(1, 2, 0).contiguous()
    ref = oracle.fwd(bits(xs), bits(wl.weight[chans]), bits(wl.bias[chans]), None,
                     bits(wl.conv_state[rows][:, chans]))
    got = outs[:, rows][:, :, chans].permute(1, 2, 0).contiguous().cpu()
    assert_bf16_close(bits(got), ref["out"], "update chain vs oracle forward")
