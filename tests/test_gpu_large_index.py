"""Activation tensors of more than 2^31 elements: every offset the kernels
form is 64-bit.  One sequence of 1 050 000 tokens by 2048 channels (2.15e9
elements, 4.3 GB per BF16 tensor; x, grad_out, out and dx together 17 GB),
channel-last and time-contiguous, forward and backward through the C ABI.
Channels are independent, so whole sampled channels -- every token, the
weight and bias sums over the full length -- are compared with the oracle
element by element: the first, middle and last channel groups, whose rows
reach the highest offsets."""

import pytest
import torch

from depthwise_causal_conv1d_channel_gb300 import _abi
import oracle
from helpers import assert_bf16_close, assert_bits_equal, assert_wgrad_close, tensor_values
from workloads import bits, device_activations

pytestmark = pytest.mark.gpu

D, T = 2048, 1_050_000
CH = [0, 1, 2, 3, 1020, 1021, 1022, 1023, 2040, 2041, 2042, 2043, 2044, 2045, 2046, 2047]


@pytest.mark.parametrize("channel_last", [True, False], ids=["channel_last", "time_contiguous"])
def test_tensors_beyond_2_31_elements(channel_last, cuda_device):
    assert D * T > 2 ** 31
    dev = cuda_device
    gen = torch.Generator().manual_seed(21)
    w = (torch.rand(D, 4, generator=gen) - 0.5).to(torch.bfloat16)
    b = ((torch.rand(D, generator=gen) - 0.5) * 0.2).to(torch.bfloat16)
    init = torch.randn(1, D, 3, generator=gen).to(torch.bfloat16)
    x = device_activations(1, D, T, dev, seed=22, channel_last=channel_last)
    g = device_activations(1, D, T, dev, seed=23, channel_last=channel_last)
    w_d, b_d, init_d = w.to(dev), b.to(dev), init.to(dev)
    out, dx = torch.empty_like(x), torch.empty_like(x)
    fin = torch.empty(1, D, 3, dtype=torch.bfloat16, device=dev)
    dinit = torch.empty_like(init_d)
    dw, db = torch.empty_like(w_d), torch.empty_like(b_d)
    ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(x, False), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    act = _abi.CCC_ACT_SILU
    assert _abi.ccc_conv1d_fwd(x, w_d, b_d, None, init_d, out, fin, act, status, stream) == _abi.CCC_OK
    assert _abi.ccc_conv1d_bwd(x, w_d, b_d, None, init_d, g, None, dx, dw, db, dinit, act, False, ws,
                               status, stream) == _abi.CCC_OK
    assert _abi.ccc_read_status(status, stream) == _abi.CCC_OK

    x_s, g_s = x[:, CH, :].cpu(), g[:, CH, :].cpu()
    ref = oracle.fwd(bits(x_s), bits(w[CH]), bits(b[CH]), None, bits(init[:, CH]), "silu")
    assert_bf16_close(bits(out[:, CH, :].cpu()), ref["out"], "out")
    assert_bits_equal(bits(fin[:, CH].cpu()), ref["final"], "final_states")
    rb = oracle.bwd(bits(x_s), bits(w[CH]), bits(g_s), bits(b[CH]), None, bits(init[:, CH]), None,
                    "silu")
    assert_bf16_close(bits(dx[:, CH, :].cpu()), rb["dx"], "dx")
    assert_bf16_close(bits(dinit[:, CH].cpu()), rb["dinit"], "dinitial_states")
    assert_wgrad_close(tensor_values(dw[CH]), rb["dw64"], rb["dw_abs"], True, "dweight")
    assert_wgrad_close(tensor_values(db[CH]), rb["db64"], rb["db_abs"], True, "dbias")
