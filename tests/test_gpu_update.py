"""GPU parity of causal_conv1d_update (the single-token decode step that
mutates the width-four state in place) against the oracle, including the
hand-off from the forward's final_states."""

import numpy as np
import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
import oracle
from helpers import assert_bf16_close, assert_bits_equal
from workloads import bits, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,D", [(4, 264), (3, 100), (1, 8), (2, 1), (256, 64), (37, 4104),
                                 (300, 1028), (129, 4096)])
@pytest.mark.parametrize("act", ["silu", None])
def test_update_parity(B, D, act, cuda_device):
    gen = torch.Generator().manual_seed(B * 7 + D)
    state = torch.randn(B, D, 3, generator=gen).to(torch.bfloat16)
    x = torch.randn(B, D, generator=gen).to(torch.bfloat16)
    w = (torch.rand(D, 4, generator=gen) - 0.5).to(torch.bfloat16)
    b = ((torch.rand(D, generator=gen) - 0.5) * 0.2).to(torch.bfloat16)
    ref = oracle.update(bits(x), bits(state), bits(w), bits(b), act)
    s_dev = state.to(cuda_device)
    out = ccc.causal_conv1d_update(x.to(cuda_device), s_dev, w.to(cuda_device), b.to(cuda_device), act)
    torch.cuda.synchronize()
    assert_bf16_close(bits(out.cpu()), ref["out"], "out")
    assert_bits_equal(bits(s_dev.cpu()), ref["state"], "state")


def test_update_strided_rows(cuda_device):
    """x and out rows with a stride larger than D (slices of wider buffers)."""
    B, D = 70, 2048
    gen = torch.Generator().manual_seed(11)
    state = torch.randn(B, D, 3, generator=gen).to(torch.bfloat16)
    xw = torch.randn(B, D + 64, generator=gen).to(torch.bfloat16)
    w = (torch.rand(D, 4, generator=gen) - 0.5).to(torch.bfloat16)
    b = ((torch.rand(D, generator=gen) - 0.5) * 0.2).to(torch.bfloat16)
    x = xw[:, 8:8 + D]
    ref = oracle.update(bits(x), bits(state), bits(w), bits(b))
    s_dev = state.to(cuda_device)
    ow = torch.zeros(B, D + 32, dtype=torch.bfloat16, device=cuda_device)
    out = ow[:, 16:16 + D]
    ccc.causal_conv1d_update(xw.to(cuda_device)[:, 8:8 + D], s_dev, w.to(cuda_device),
                             b.to(cuda_device), out=out)
    torch.cuda.synchronize()
    assert_bf16_close(bits(out.cpu()), ref["out"], "out")
    assert_bits_equal(bits(s_dev.cpu()), ref["state"], "state")
    assert not ow[:, :16].any() and not ow[:, 16 + D:].any()


def test_update_fp32_weight_no_bias(cuda_device):
    B, D = 8, 40
    gen = torch.Generator().manual_seed(3)
    state = torch.randn(B, D, 3, generator=gen).to(torch.bfloat16)
    x = torch.randn(B, D, generator=gen).to(torch.bfloat16)
    w = torch.rand(D, 4, generator=gen) - 0.5
    ref = oracle.update(bits(x), bits(state), w.numpy(), None)
    s_dev = state.to(cuda_device)
    out = ccc.causal_conv1d_update(x.to(cuda_device), s_dev, w.to(cuda_device))
    torch.cuda.synchronize()
    assert_bf16_close(bits(out.cpu()), ref["out"], "out")
    assert_bits_equal(bits(s_dev.cpu()), ref["state"], "state")


def test_forward_final_state_feeds_update_chain(cuda_device):
    """Prefill with the forward, then decode token by token: equals one
    forward over the whole sequence (cuDNN page: final_states pass directly to
    causal_conv1d_update, no layout conversion)."""
    B, D, T, steps = 3, 136, 40, 25
    full = make_inputs(B, D, T + steps, seed=17, initial_states=True)
    d = full.to(cuda_device)
    out_pre, state = ccc.causal_conv1d(d.x[:, :, :T], d.weight, d.bias,
                                       initial_states=d.initial_states, return_final_states=True)
    outs = []
    for s in range(steps):
        xt = d.x[:, :, T + s].contiguous()
        outs.append(ccc.causal_conv1d_update(xt, state, d.weight, d.bias))
    torch.cuda.synchronize()
    ref = oracle.fwd(bits(full.x), bits(full.weight), bits(full.bias), None, bits(full.initial_states))
    assert_bf16_close(bits(out_pre.cpu()), np.ascontiguousarray(ref["out"][:, :, :T]), "prefill")
    chain = torch.stack(outs, dim=2).cpu()
    assert_bf16_close(bits(chain), np.ascontiguousarray(ref["out"][:, :, T:]), "decode chain")
    assert_bits_equal(bits(state.cpu()), ref["final"], "state after chain")
    # the GPU forward and the GPU update chain evaluate the same FMA sequence
    gpu_full = ccc.causal_conv1d(d.x, d.weight, d.bias, initial_states=d.initial_states)
    assert torch.equal(gpu_full[:, :, T:].contiguous().view(torch.int16).cpu(),
                       chain.contiguous().view(torch.int16))


# ---- several tokens per row: x [B, D, L] -------------------------------------

def _multi_inputs(B, D, L, seed, channel_last=True, weight_dtype=torch.bfloat16, bias=True):
    """Inputs of a multi-token update, as a forward problem over the L tokens
    (initial_states = the state before the update)."""
    return make_inputs(B, D, L, seed=seed, channel_last=channel_last, initial_states=True,
                       weight_dtype=weight_dtype, bias=bias)


@pytest.mark.parametrize("B,D,L", [(3, 264, 5), (2, 100, 7), (4, 4096, 3), (1, 8, 1), (5, 36, 64),
                                   (2, 1, 4), (2, 512, 4), (3, 520, 8), (2, 264, 9), (1, 256, 2)])
@pytest.mark.parametrize("act", ["silu", None])
def test_multi_token_update_parity(B, D, L, act, cuda_device):
    """Each row's L tokens in one call: out equals the oracle's forward over
    them with the old state as initial state; the new state equals its final
    state bitwise."""
    inp = _multi_inputs(B, D, L, seed=B * 31 + D + L)
    ref = oracle.fwd(bits(inp.x), bits(inp.weight), bits(inp.bias), None,
                     bits(inp.initial_states), act)
    d = inp.to(cuda_device)
    state = d.initial_states.clone()
    out = ccc.causal_conv1d_update(d.x, state, d.weight, d.bias, act)
    torch.cuda.synchronize()
    assert out.shape == (B, D, L) and (D == 1 or out.stride(1) == 1)
    assert_bf16_close(bits(out.cpu()), ref["out"], "out")
    assert_bits_equal(bits(state.cpu()), ref["final"], "state")


@pytest.mark.parametrize("wdtype", [torch.bfloat16, torch.float32])
def test_multi_token_update_equals_forward_bitwise(wdtype, cuda_device):
    """The update over L tokens and the forward over the same tokens evaluate
    the same operations in the same order: bitwise equal outputs and state."""
    B, D, L = 3, 520, 11
    inp = _multi_inputs(B, D, L, seed=7, weight_dtype=wdtype, bias=wdtype == torch.bfloat16)
    d = inp.to(cuda_device)
    fwd_out, fin = ccc.causal_conv1d(d.x, d.weight, d.bias, initial_states=d.initial_states,
                                     return_final_states=True)
    state = d.initial_states.clone()
    out = ccc.causal_conv1d_update(d.x, state, d.weight, d.bias)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), fwd_out.view(torch.int16))
    assert torch.equal(state.view(torch.int16), fin.view(torch.int16))


def test_multi_token_update_layouts_and_chunks(cuda_device):
    """Time-contiguous x (restrided by the wrapper), a strided token axis, and
    a sequence fed in chunks of 5, 1, 0 and 9 tokens: all equal one forward."""
    B, D, L = 2, 1032, 15
    inp = _multi_inputs(B, D, L, seed=3, channel_last=False)
    ref = oracle.fwd(bits(inp.x), bits(inp.weight), bits(inp.bias), None,
                     bits(inp.initial_states))
    d = inp.to(cuda_device)
    assert d.x.stride(2) == 1  # time-contiguous
    state = d.initial_states.clone()
    out = ccc.causal_conv1d_update(d.x, state, d.weight, d.bias)
    torch.cuda.synchronize()
    assert_bf16_close(bits(out.cpu()), ref["out"], "out (time-contiguous x)")
    assert_bits_equal(bits(state.cpu()), ref["final"], "state (time-contiguous x)")
    # channel-last storage with every other token: token stride 2 * D
    wide = torch.zeros(B, 2 * L, D, dtype=torch.bfloat16, device=cuda_device)
    wide[:, ::2] = inp.x.transpose(1, 2).to(cuda_device)
    xs = wide[:, ::2].transpose(1, 2)
    assert xs.stride() == (2 * L * D, 1, 2 * D)
    state = d.initial_states.clone()
    outs = []
    for lo, hi in [(0, 5), (5, 6), (6, 6), (6, 15)]:
        outs.append(ccc.causal_conv1d_update(xs[:, :, lo:hi], state, d.weight, d.bias))
    torch.cuda.synchronize()
    chunked = torch.cat(outs, dim=2).cpu()
    assert_bf16_close(bits(chunked), ref["out"], "out (chunks)")
    assert_bits_equal(bits(state.cpu()), ref["final"], "state (chunks)")


def test_multi_token_update_in_place(cuda_device):
    """out may be x itself: the update then overwrites the tokens with the outputs."""
    B, D, L = 4, 256, 6
    inp = _multi_inputs(B, D, L, seed=19)
    ref = oracle.fwd(bits(inp.x), bits(inp.weight), bits(inp.bias), None,
                     bits(inp.initial_states))
    d = inp.to(cuda_device)
    x = d.x.transpose(1, 2).contiguous().transpose(1, 2)  # own copy, channel-last
    state = d.initial_states.clone()
    out = ccc.causal_conv1d_update(x, state, d.weight, d.bias, out=x)
    torch.cuda.synchronize()
    assert out.data_ptr() == x.data_ptr()
    assert_bf16_close(bits(x.cpu()), ref["out"], "in-place out")
    assert_bits_equal(bits(state.cpu()), ref["final"], "state")
