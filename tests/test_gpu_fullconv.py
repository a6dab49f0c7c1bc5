"""GPU parity of the full-channel dilated causal conv1d (POPCORNBENCH conv1d
page) on the tensor cores, against the fp64 oracle on the same seeded inputs.

Tolerance (helpers.assert_fullconv_close): |gpu - ref| <= 1e-3 * sum|terms| +
2^-8 * |ref|.  Cases span several output tiles along tokens and channels with
ragged tails (T, Cout, and Cin not multiples of the 128 / 256 / 64 tile),
receptive fields longer than the sequence, receptive fields up to the widest
x slice the persistent kernel holds and beyond it (the per-tap kernel), K = 1,
calls of hundreds of tiles (several per CTA, whole and half tiles),
FP32 weights and biases
(the pack rounds the weight to BF16; the oracle takes the rounded weight),
strided inputs, and the full-size workload on sampled output channels.
"""

import numpy as np
import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
import oracle
from depthwise_causal_conv1d_channel_gb300 import _abi
from helpers import assert_fullconv_close
from workloads import bits, fullconv_dilated, fullconv_inputs

pytestmark = pytest.mark.gpu


def _weight_bits_as_packed(w):
    """The oracle's view of the packed weight: BF16 bits of W (FP32 rounded to
    nearest even by the oracle's own rounding)."""
    if w.dtype == torch.float32:
        return oracle.bf16_encode(w.double().numpy())
    return bits(w)


def _bias_np(b):
    if b is None:
        return None
    return b.numpy() if b.dtype == torch.float32 else bits(b)


def gpu_fullconv(inp, device):
    d = inp.to(device)
    out = ccc.full_causal_conv1d(d.x, d.weight, d.bias, inp.dilation)
    ccc.check_status(device)
    torch.cuda.synchronize()
    return out


CASES = [
    # (B, Cin, Cout, T, K, dilation, options)
    (2, 64, 256, 300, 4, 2, {}),
    (1, 136, 264, 129, 3, 5, dict(bias_dtype=torch.float32)),
    (3, 8, 8, 7, 4, 40, {}),                       # receptive field far longer than T
    (2, 256, 512, 256, 1, 1, dict(bias=False)),    # K = 1: a plain matrix product
    (1, 72, 40, 1000, 2, 97, dict(weight_dtype=torch.float32, bias=False)),
    (2, 512, 128, 384, 4, 1, {}),
    (1, 128, 256, 700, 5, 64, {}),                 # receptive field 256: the widest x slice
    (2, 64, 136, 600, 3, 200, {}),                 # receptive field 400: one x slice per tap
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}Ci{c[1]}Co{c[2]}T{c[3]}K{c[4]}d{c[5]}")
def test_fullconv_parity(case, cuda_device):
    B, Cin, Cout, T, K, dil, opts = case
    inp = fullconv_inputs(B, Cin, Cout, T, K, dil, seed=B + Cin + T, **opts)
    out = gpu_fullconv(inp, cuda_device)
    assert out.shape == (B, Cout, T) and out.stride(1) == 1
    ref = oracle.fullconv(bits(inp.x), _weight_bits_as_packed(inp.weight), _bias_np(inp.bias), dil)
    assert_fullconv_close(bits(out.cpu()), ref["out64"], ref["abs_sum"])


SCHEDULE_CASES = [
    # (B, Cin, Cout, T, K, dilation): many 256 x 256 tiles per call, so that a
    # CTA takes several of them in turn
    (1, 64, 256, 256 * 250, 4, 2),    # 250 tiles: the last wave is more than half full
    (2, 64, 256, 25500, 3, 7),        # 200 tiles: one wave, then halves (ragged token tail)
    (1, 128, 512, 256 * 160, 2, 1),   # 320 tiles: two waves, then halves
]


@pytest.mark.parametrize("case", SCHEDULE_CASES, ids=lambda c: f"B{c[0]}Co{c[2]}T{c[3]}")
def test_fullconv_persistent_schedule(case, cuda_device):
    """Calls of hundreds of tiles, which each CTA of the persistent kernel
    walks several of (whole tiles and, where the last wave is at most half
    full, half tiles).  Output channels are independent given x, so a sample
    of whole channels from every channel tile is checked element by element."""
    B, Cin, Cout, T, K, dil = case
    inp = fullconv_inputs(B, Cin, Cout, T, K, dil, seed=T + Cout)
    out = gpu_fullconv(inp, cuda_device).cpu()
    chans = sorted({c for base in range(0, Cout, 256) for c in (base, base + 1, base + 130, base + 255)
                    if c < Cout})
    ref = oracle.fullconv(bits(inp.x), bits(inp.weight[chans]), bits(inp.bias[chans]), dil)
    assert_fullconv_close(bits(out[:, chans]), ref["out64"], ref["abs_sum"])


def test_fullconv_pack_weight_is_tap_major_and_rounds_to_bf16(cuda_device):
    w32 = torch.randn(24, 16, 3, generator=torch.Generator().manual_seed(3))
    packed = ccc.pack_full_conv_weight(w32.to(cuda_device)).cpu()
    assert packed.shape == (3, 24, 16)
    ref = oracle.bf16_encode(w32.double().numpy()).transpose(2, 0, 1)
    assert np.array_equal(bits(packed), ref)
    # a BF16 weight given as a strided view is copied bitwise
    wb = torch.randn(16, 3, 24, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    view = wb.to(cuda_device).permute(2, 0, 1)  # [24, 16, 3], non-contiguous
    packed = ccc.pack_full_conv_weight(view).cpu()
    assert np.array_equal(bits(packed), bits(wb.permute(2, 0, 1)).transpose(2, 0, 1))


def test_fullconv_strided_rows_and_repeatable(cuda_device):
    """x and out as views with token strides larger than the channel count;
    two calls give bitwise equal results."""
    B, Cin, Cout, T, K, dil = 2, 64, 96, 200, 3, 3
    inp = fullconv_inputs(B, Cin, Cout, T, K, dil, seed=17)
    d = inp.to(cuda_device)
    xs = torch.zeros(B, T, Cin + 16, dtype=torch.bfloat16, device=cuda_device)
    xs[:, :, :Cin] = d.x.transpose(1, 2)
    x_view = xs[:, :, :Cin].transpose(1, 2)
    packed = ccc.pack_full_conv_weight(d.weight)
    big = torch.full((B, T, Cout + 24), 7.0, dtype=torch.bfloat16, device=cuda_device)
    out_view = big[:, :, :Cout].transpose(1, 2)
    stream = torch.cuda.current_stream(cuda_device)
    assert _abi.ccc_fullconv1d_fwd(x_view, packed, d.bias, dil, out_view, None, stream) == 0
    first = out_view.clone()
    assert _abi.ccc_fullconv1d_fwd(x_view, packed, d.bias, dil, out_view, None, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(first, out_view)
    assert torch.all(big[:, :, Cout:] == 7.0)  # the padding columns are untouched
    ref = oracle.fullconv(bits(inp.x), bits(inp.weight), bits(inp.bias), dil)
    assert_fullconv_close(bits(out_view.cpu()), ref["out64"], ref["abs_sum"])


def test_fullconv_workload_sampled_channels(cuda_device):
    """The measured workload (8 x 4096 tokens, 1024 -> 1024 channels, K 4,
    dilation 2) at full size; output channels are independent given x, so
    whole sampled channels of sampled rows are checked element by element."""
    inp = fullconv_dilated()
    out = gpu_fullconv(inp, cuda_device).cpu()
    # row 7 holds the tiles that the last wave cuts into halves of 128 tokens
    for b in (0, 5, 7):
        chans = [0, 1, 255, 256, 511, 700, 1023]
        xb = bits(inp.x[b:b + 1])
        ref = oracle.fullconv(xb, bits(inp.weight[chans]), bits(inp.bias[chans]), inp.dilation)
        assert_fullconv_close(bits(out[b:b + 1, chans]), ref["out64"], ref["abs_sum"])


def test_fullconv_host_rejections(cuda_device):
    inp = fullconv_inputs(1, 64, 64, 32, 2, 1, seed=1)
    d = inp.to(cuda_device)
    packed = ccc.pack_full_conv_weight(d.weight)
    stream = torch.cuda.current_stream(cuda_device)
    out = torch.empty(1, 32, 64, dtype=torch.bfloat16, device=cuda_device).transpose(1, 2)
    # time-contiguous x is not read by the kernel (the Python call restrides it)
    xt = d.x.contiguous()
    assert _abi.ccc_fullconv1d_fwd(xt, packed, d.bias, 1, out, None, stream) == _abi.CCC_ERR_UNSUPPORTED
    assert _abi.ccc_fullconv1d_fwd(d.x, packed, d.bias, 0, out, None, stream) == _abi.CCC_ERR_INVALID_ARG
    # out on top of x
    assert _abi.ccc_fullconv1d_fwd(d.x, packed, d.bias, 1, d.x, None, stream) == _abi.CCC_ERR_ALIAS
    # the Python call restrides a contiguous x and gives the same result
    a = ccc.full_causal_conv1d(xt, packed_weight=packed, bias=d.bias)
    b = ccc.full_causal_conv1d(d.x, packed_weight=packed, bias=d.bias)
    assert torch.equal(a, b)
