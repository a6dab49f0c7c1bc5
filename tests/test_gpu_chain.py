"""Forward calls chained on one stream, each reading what the one before it
wrote.

Every depthwise kernel is launched as a programmatic dependent of the kernel
before it, and the dense channel-last forward prefetches its first input rows
into L2 before it waits for that kernel to finish.  A prefetch only moves
lines into L2, so each call must still compute on the finished output of the
call before it.  Here every step writes a fresh buffer that held a poison
pattern until then; each step is checked against the oracle applied to the
input it read (the previous step's output as stored), so a step that read
stale or unfinished data shows up as a mismatch.
"""

import dataclasses

import pytest
import torch

from depthwise_causal_conv1d_channel_gb300 import _abi
import oracle
from helpers import assert_bf16_close, assert_bits_equal, oracle_fwd
from workloads import bits, make_inputs, seq_ids

pytestmark = pytest.mark.gpu

STEPS = 6
POISON_BITS = 0x7FC1  # a BF16 NaN


CASES = {
    # dense channel-last (the forward that prefetches before its wait)
    "dense": dict(B=4, D=512, T=600, kw=dict(initial_states=True)),
    # short ranges: 3-token ring groups
    "dense_short": dict(B=8, D=256, T=96, kw=dict(initial_states=True)),
    # packed sequences (no prefetch before the wait)
    "packed": dict(B=1, D=256, T=1000, kw=dict(initial_states=True, lengths=[1, 300, 17, 500, 182])),
    # per-token sequence ids (the id instance prefetches too)
    "seq_idx": dict(B=3, D=256, T=700, kw=dict(), ids=True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_chain_reads_previous_output(name, cuda_device):
    case = CASES[name]
    inp = make_inputs(case["B"], case["D"], case["T"], seed=23, **case["kw"])
    ids = seq_ids(case["B"], case["T"], seed=5, max_run=64) if case.get("ids") else None
    d = inp.to(cuda_device)
    ids_d = ids.to(cuda_device) if ids is not None else None
    act = _abi.CCC_ACT_SILU
    # buffers 1..STEPS start as poison; step k reads buffer k and writes k + 1
    bufs = [d.x] + [torch.empty_like(d.x) for _ in range(STEPS)]
    for b in bufs[1:]:
        b.view(torch.int16).fill_(POISON_BITS)
    fins = [torch.empty_like(d.initial_states) if d.initial_states is not None else None
            for _ in range(STEPS)]
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    stream = torch.cuda.current_stream(cuda_device)
    torch.cuda.synchronize(cuda_device)
    for k in range(STEPS):
        rc = _abi.ccc_conv1d_fwd(bufs[k], d.weight, d.bias, d.cu_seqlens, d.initial_states,
                                 bufs[k + 1], fins[k], act, status, stream, seq_idx=ids_d)
        assert rc == _abi.CCC_OK
    assert _abi.ccc_read_status(status, stream) == _abi.CCC_OK
    torch.cuda.synchronize(cuda_device)
    for k in range(STEPS):
        src = bufs[k].cpu()
        step = dataclasses.replace(inp, x=src)
        ref = oracle_fwd(step) if ids is None else oracle_fwd_ids(step, ids)
        assert_bf16_close(bits(bufs[k + 1].cpu()), ref["out"], f"step {k} out")
        if fins[k] is not None:
            assert_bits_equal(bits(fins[k].cpu()), ref["final"], f"step {k} final")


def oracle_fwd_ids(inp, ids):
    return oracle.fwd(bits(inp.x), bits(inp.weight), bits(inp.bias), None, None, inp.activation,
                      seq_idx=ids.numpy())
