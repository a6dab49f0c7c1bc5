"""Filter widths W = 2 and 3 (the page's tensors are weight[D, W] and states
[., D, W - 1]; its optimized route is W = 4).  The kernels embed a width-W
filter in width four with leading zero taps: parity against the oracle's
width-W forward, backward and update, on the vector and scalar paths, dense
and packed, both layouts."""

import numpy as np
import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
import oracle
from helpers import assert_bf16_close, assert_bits_equal, assert_wgrad_close, tensor_values
from workloads import bits, from_bits

pytestmark = pytest.mark.gpu


def _inputs(B, D, T, W, seed, lengths=None, channel_last=True, wdtype=torch.bfloat16, bias=True):
    gen = torch.Generator().manual_seed(seed)
    S = B if lengths is None else len(lengths)
    shape = (B, T, D) if channel_last else (B, D, T)
    x = torch.randn(shape, generator=gen).to(torch.bfloat16)
    g = torch.randn(shape, generator=gen).to(torch.bfloat16)
    if channel_last:
        x, g = x.transpose(1, 2), g.transpose(1, 2)
    w = (torch.rand(D, W, generator=gen) - 0.5)
    w = w if wdtype == torch.float32 else w.to(torch.bfloat16)
    b = ((torch.rand(D, generator=gen) - 0.5) * 0.2).to(torch.bfloat16) if bias else None
    init = torch.randn(S, D, W - 1, generator=gen).to(torch.bfloat16)
    gf = torch.randn(S, D, W - 1, generator=gen).to(torch.bfloat16)
    cu = None
    if lengths is not None:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return x, g, w, b, init, gf, cu


def _to(t, dev, channel_last):
    if t is None:
        return None
    if channel_last and t.dim() == 3 and t.shape[2] > 3:
        return t.transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    return t.to(dev)


CASES = [
    # (B, D, T, lengths, channel_last, wdtype, bias) -- D multiple of 8 / 4 / odd, dense / packed
    (2, 264, 70, None, True, torch.bfloat16, True),
    (3, 100, 33, None, True, torch.bfloat16, True),
    (2, 37, 21, None, True, torch.bfloat16, False),
    (1, 136, 0, [7, 1, 40, 2], True, torch.float32, False),
    (2, 48, 50, None, False, torch.bfloat16, True),
    (1, 24, 0, [5, 9, 1], False, torch.bfloat16, True),
    (2, 16, 264, None, False, torch.bfloat16, True),   # time-contiguous, 8 tokens a lane
    (1, 2048, 20000, None, True, torch.float32, False),  # long ranges: the 8-channel backward
    (1, 1024, 40000, None, True, torch.bfloat16, True),
]


@pytest.mark.parametrize("W", [2, 3])
@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_width_parity(W, case, cuda_device):
    B, D, T, lengths, cl, wdtype, with_bias = case
    if lengths is not None:
        T = sum(lengths)
    x, g, w, b, init, gf, cu = _inputs(B, D, T, W, seed=W * 100 + D + T, lengths=lengths,
                                       channel_last=cl, wdtype=wdtype, bias=with_bias)
    wbits = w.numpy() if wdtype == torch.float32 else bits(w)
    cun = None if cu is None else cu.numpy()
    rf = oracle.fwd(bits(x), wbits, bits(b), cun, bits(init))
    rb = oracle.bwd(bits(x), wbits, bits(g), bits(b), cun, bits(init), bits(gf))

    dx_, dw_ = _to(x, cuda_device, cl).detach().requires_grad_(True), w.to(cuda_device).requires_grad_(True)
    db_ = b.to(cuda_device).requires_grad_(True) if b is not None else None
    di_ = init.to(cuda_device).requires_grad_(True)
    out, fin = ccc.causal_conv1d(dx_, dw_, db_, cu_seqlens=None if cu is None else cu.to(cuda_device),
                                 initial_states=di_, return_final_states=True)
    assert fin.shape == (init.shape[0], D, W - 1)
    torch.autograd.backward([out, fin], [_to(g, cuda_device, cl), gf.to(cuda_device)])
    ccc.check_status(cuda_device)
    torch.cuda.synchronize()
    assert_bf16_close(bits(out.detach().cpu()), rf["out"], "out")
    assert_bits_equal(bits(fin.detach().cpu()), rf["final"], "final")
    assert_bf16_close(bits(dx_.grad.cpu()), rb["dx"], "dx")
    assert_bf16_close(bits(di_.grad.cpu()), rb["dinit"], "dinit")
    assert_wgrad_close(tensor_values(dw_.grad), rb["dw64"], rb["dw_abs"], wdtype == torch.bfloat16,
                       "dweight")
    if b is not None:
        assert_wgrad_close(tensor_values(db_.grad), rb["db64"], rb["db_abs"], True, "dbias")


@pytest.mark.parametrize("W", [2, 3])
@pytest.mark.parametrize("B,D,L", [(4, 264, 1), (3, 4096, 1), (2, 100, 6), (5, 37, 3)])
def test_width_update_parity(W, B, D, L, cuda_device):
    """Decode update with a width-W state [B, D, W - 1]: equals the oracle's
    width-W forward over the L tokens, state bitwise."""
    x, _, w, b, init, _, _ = _inputs(B, D, L, W, seed=W * 7 + D + L)
    rf = oracle.fwd(bits(x), bits(w), bits(b), None, bits(init))
    state = init.to(cuda_device).clone()
    xs = _to(x, cuda_device, True) if L > 1 else x[:, :, 0].contiguous().to(cuda_device)
    out = ccc.causal_conv1d_update(xs, state, w.to(cuda_device), b.to(cuda_device))
    torch.cuda.synchronize()
    got = out.cpu() if L > 1 else out.cpu()[:, :, None]
    assert_bf16_close(bits(got), rf["out"], "out")
    assert_bits_equal(bits(state.cpu()), rf["final"], "state")


def test_width_mismatched_state_is_rejected(cuda_device):
    x = torch.zeros(1, 16, 8, dtype=torch.bfloat16, device=cuda_device)
    w = torch.zeros(16, 3, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError):
        ccc.causal_conv1d(x, w, initial_states=torch.zeros(1, 16, 3, dtype=torch.bfloat16,
                                                           device=cuda_device))
    with pytest.raises(NotImplementedError):
        ccc.causal_conv1d(x, torch.zeros(16, 5, dtype=torch.bfloat16, device=cuda_device))
