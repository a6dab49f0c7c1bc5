"""Device-side validation of cu_seqlens without a device trap.

The cuDNN page executes a device trap on malformed packed metadata; here every
thread block validates the offsets, skips its writes and records
CCC_ERR_BAD_CU_SEQLENS in the status word.  These tests feed each malformed
class from the page (first offset non-zero, last offset != token total,
non-increasing offsets, empty sequence), read the status, and check that the
CUDA context stays usable by running a well-formed call afterwards.  The
kernels read nothing out of bounds on malformed input because no block touches
memory before its validation passes.
"""

import pytest
import torch

import depthwise_causal_conv1d_channel_gb300 as ccc
from conftest import golden
from depthwise_causal_conv1d_channel_gb300 import _abi
from helpers import assert_bf16_close, oracle_fwd
from workloads import bits, make_inputs

pytestmark = pytest.mark.gpu


def _bad_cases():
    return [c for c in golden("cu_seqlens_cases.json")["cases"] if not c["valid"]]


@pytest.mark.parametrize("case", _bad_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("cl", [True, False])
def test_malformed_cu_seqlens_sets_status(case, cl, cuda_device):
    total = case["total"]
    D = 16
    inp = make_inputs(1, D, total, channel_last=cl, seed=2, grad=True)
    d = inp.to(cuda_device)
    cu = torch.tensor(case["cu_seqlens"], dtype=torch.int32, device=cuda_device)
    N = cu.numel() - 1
    init = torch.zeros(N, D, 3, dtype=torch.bfloat16, device=cuda_device)
    st = ccc.status_word(cuda_device)
    ccc.check_status(cuda_device)  # clear
    out = torch.empty_like(d.x)
    fin = torch.empty(N, D, 3, dtype=torch.bfloat16, device=cuda_device)
    rc = _abi.ccc_conv1d_fwd(d.x, d.weight, d.bias, cu, init, out, fin, 1, st,
                             torch.cuda.current_stream())
    assert rc == _abi.CCC_OK  # the host does not read cu_seqlens
    assert _abi.ccc_read_status(st, torch.cuda.current_stream()) == _abi.CCC_ERR_BAD_CU_SEQLENS
    # backward, deterministic flag on and off
    for det in (False, True):
        dx = torch.empty_like(d.x)
        dw = torch.empty_like(d.weight)
        ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(d.x, det), dtype=torch.uint8,
                         device=cuda_device)
        rc = _abi.ccc_conv1d_bwd(d.x, d.weight, None, cu, init, d.g, None, dx, dw, None, None, 1,
                                 det, ws, st, torch.cuda.current_stream())
        assert rc == _abi.CCC_OK
        assert _abi.ccc_read_status(st, torch.cuda.current_stream()) == _abi.CCC_ERR_BAD_CU_SEQLENS
    # the Python API surfaces it on check_status
    ccc.causal_conv1d(d.x, d.weight, d.bias, cu_seqlens=cu)
    with pytest.raises(ccc.Conv1dError):
        ccc.check_status(cuda_device)
    # the context is still usable: a well-formed call succeeds and is correct
    good = make_inputs(1, D, 12, channel_last=cl, seed=3, lengths=[5, 7])
    g = good.to(cuda_device)
    out = ccc.causal_conv1d(g.x, g.weight, g.bias, cu_seqlens=g.cu_seqlens)
    ccc.check_status(cuda_device)
    assert_bf16_close(bits(out.cpu()), oracle_fwd(good)["out"], "out after error")


def test_host_side_errors_raise_python_exceptions(cuda_device):
    inp = make_inputs(2, 16, 10, seed=1, initial_states=True)
    d = inp.to(cuda_device)
    with pytest.raises(NotImplementedError):   # FP32 weight with bias declines
        ccc.causal_conv1d(d.x, d.weight.float(), d.bias)
    with pytest.raises(NotImplementedError):   # width outside 2..4
        ccc.causal_conv1d(d.x, torch.zeros(16, 5, dtype=torch.bfloat16, device=cuda_device))
    with pytest.raises(ValueError):            # final_states_out aliasing x
        ccc.causal_conv1d(d.x, d.weight, d.bias, initial_states=d.initial_states,
                          final_states_out=d.x.transpose(1, 2).reshape(-1)[: 2 * 16 * 3].view(2, 16, 3))
