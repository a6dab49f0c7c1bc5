"""ccc_conv1d_bwd_noalloc: the backward for callers that cannot allocate device
memory (a host program that owns all device memory and forbids allocation
while it runs, so it cannot hand over the workspace ccc_conv1d_bwd needs).
The entry point uses the library's built-in scratch instead.

Checked through the C ABI against ccc_conv1d_bwd with a caller workspace, on
two calls in a row (the second finds the scratch holding the first call's
contents): both calls run the same kernels on the same grid and add the same
partial rows in the same fixed order, so every output must be bitwise equal
to the workspace backward's; and against the oracle, with the tolerances the
other parity tests use.  The cases reach the channel-last kernels, both
time-contiguous kernels (one row a warp, and two rows a warp for rows of 4096
tokens or more), the packed route and the empty sequence (which zeroes the
first partial row itself); plus the size limit.  This file is collected last
on purpose.
"""

import pytest
import torch

from depthwise_causal_conv1d_channel_gb300 import _abi
from helpers import assert_bf16_close, assert_wgrad_close, oracle_bwd, tensor_values
from workloads import bits, make_inputs

pytestmark = pytest.mark.gpu


def _outputs(d):
    dx = torch.empty_like(d.x)
    dw = torch.empty_like(d.weight)
    db = torch.empty_like(d.bias) if d.bias is not None else None
    dinit = torch.empty_like(d.initial_states)
    return dx, dw, db, dinit


CASES = [
    dict(B=2, D=264, T=300, lengths=None, det=False, channel_last=True),
    dict(B=1, D=512, T=1200, lengths=[5, 300, 1, 800, 94], det=True, channel_last=True),
    dict(B=3, D=40, T=256, lengths=None, det=False, channel_last=False),
    dict(B=2, D=64, T=4096, lengths=None, det=True, channel_last=False),
    dict(B=2, D=64, T=0, lengths=None, det=False, channel_last=True),
]
IDS = ["dense-default", "packed-deterministic", "time-contiguous-row-a-warp",
       "time-contiguous-two-rows-a-warp-deterministic", "empty-sequence"]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_noalloc_backward_matches_workspace_backward_twice(case, cuda_device):
    det = case["det"]
    inp = make_inputs(case["B"], case["D"], case["T"], seed=31, lengths=case["lengths"],
                      initial_states=True, grad=True, dfinal_states=True, bias=not det,
                      weight_dtype=torch.float32 if det else torch.bfloat16,
                      channel_last=case["channel_last"])
    d = inp.to(cuda_device)
    stream = torch.cuda.current_stream(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)

    # the existing entry point, with a workspace the caller allocates
    rdx, rdw, rdb, rdi = _outputs(d)
    ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(d.x, det), dtype=torch.uint8,
                     device=cuda_device)
    assert _abi.ccc_conv1d_bwd(d.x, d.weight, d.bias, d.cu_seqlens, d.initial_states, d.g,
                               d.dfinal_states, rdx, rdw, rdb, rdi, _abi.CCC_ACT_SILU, det, ws,
                               status, stream) == _abi.CCC_OK
    assert _abi.ccc_read_status(status, stream) == _abi.CCC_OK
    ref = oracle_bwd(inp)
    bf16_w = inp.weight.dtype == torch.bfloat16

    for _ in range(2):
        dx, dw, db, dinit = _outputs(d)
        rc = _abi.ccc_conv1d_bwd_noalloc(d.x, d.weight, d.bias, d.cu_seqlens, d.initial_states,
                                         d.g, d.dfinal_states, dx, dw, db, dinit,
                                         _abi.CCC_ACT_SILU, det, status, stream)
        assert rc == _abi.CCC_OK, _abi.status_string(rc)
        assert _abi.ccc_read_status(status, stream) == _abi.CCC_OK
        # against the existing entry point: same kernels, same fixed-order sums
        assert torch.equal(dx, rdx), "dx differs from the workspace backward"
        assert torch.equal(dinit, rdi), "dinitial_states differ from the workspace backward"
        assert torch.equal(dw, rdw), "dweight differs from the workspace backward"
        if db is not None:
            assert torch.equal(db, rdb), "dbias differs from the workspace backward"
        # and against the oracle
        assert_bf16_close(bits(dx), ref["dx"], "dx vs oracle")
        assert_bf16_close(bits(dinit), ref["dinit"], "dinit vs oracle")
        assert_wgrad_close(tensor_values(dw), ref["dw64"], ref["dw_abs"], bf16_w, "dweight vs oracle")
        if db is not None:
            assert_wgrad_close(tensor_values(db), ref["db64"], ref["db_abs"], True, "dbias vs oracle")


def test_noalloc_rejects_problems_beyond_the_scratch(cuda_device):
    # at least one row of D * 5 FP32 partial sums: 262144 channels need 5 MiB > 4 MiB
    D = 262144
    x = torch.zeros(1, 1, D, dtype=torch.bfloat16, device=cuda_device).transpose(1, 2)
    assert _abi.ccc_conv1d_bwd_workspace_size(x, False) > 4 << 20
    w = torch.zeros(D, 4, dtype=torch.bfloat16, device=cuda_device)
    b = torch.zeros(D, dtype=torch.bfloat16, device=cuda_device)
    g = torch.zeros_like(x)
    dx, dw, db = torch.empty_like(x), torch.empty_like(w), torch.empty_like(b)
    rc = _abi.ccc_conv1d_bwd_noalloc(x, w, b, None, None, g, None, dx, dw, db, None,
                                     _abi.CCC_ACT_SILU, False, None,
                                     torch.cuda.current_stream(cuda_device))
    assert rc == _abi.CCC_ERR_SCRATCH_LIMIT
    assert "scratch" in _abi.status_string(rc)
