"""The C-ABI calls inside CUDA graphs.

Every call is capturable: the host checks need no device data, nothing is
allocated or synchronised inside a call, and the kernels are launched as
programmatic dependents of one another, which a graph keeps.  A replayed graph
must give bitwise the results of the same calls made eagerly, and the
oracle's results within the usual tolerances.  The device-side cu_seqlens
validation works inside a graph too: the offsets are read by the kernels, so
a replay over offsets rewritten in place reports through the status word.
"""

import pytest
import torch

from depthwise_causal_conv1d_channel_gb300 import _abi
import oracle
from helpers import (assert_bf16_close, assert_bits_equal, assert_wgrad_close, oracle_bwd,
                     oracle_fwd, tensor_values)
from workloads import bits, make_inputs

pytestmark = pytest.mark.gpu

POISON = -12345.0  # written into every output before a replay


class Call:
    """Preallocated buffers of one forward + backward through the C ABI."""

    def __init__(self, inp, device, deterministic):
        d = inp.to(device)
        self.d = d
        self.det = deterministic
        S = inp.n_seq
        D, W = d.x.shape[1], d.weight.shape[1]
        self.act = _abi.CCC_ACT_SILU if inp.activation == "silu" else _abi.CCC_ACT_NONE
        self.out = torch.empty_like(d.x)
        self.dx = torch.empty_like(d.x)
        self.fin = (torch.empty(S, D, W - 1, dtype=torch.bfloat16, device=device)
                    if d.initial_states is not None else None)
        self.dinit = torch.empty_like(d.initial_states) if d.initial_states is not None else None
        self.dw = torch.empty_like(d.weight)
        self.db = torch.empty_like(d.bias) if d.bias is not None else None
        self.ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(d.x, deterministic),
                              dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def outputs(self):
        return [t for t in (self.out, self.fin, self.dx, self.dw, self.db, self.dinit) if t is not None]

    def launch(self, stream):
        d = self.d
        assert _abi.ccc_conv1d_fwd(d.x, d.weight, d.bias, d.cu_seqlens, d.initial_states, self.out,
                                   self.fin, self.act, self.status, stream) == _abi.CCC_OK
        assert _abi.ccc_conv1d_bwd(d.x, d.weight, d.bias, d.cu_seqlens, d.initial_states, d.g,
                                   d.dfinal_states, self.dx, self.dw, self.db, self.dinit, self.act,
                                   self.det, self.ws, self.status, stream) == _abi.CCC_OK

    def read_status(self, stream):
        return _abi.ccc_read_status(self.status, stream)


def capture(fn, device):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn(s)
    torch.cuda.synchronize()
    return g


CASES = [
    # channel-last, four channels a thread, state in and out
    ("dense_channel_last", dict(B=2, D=264, T=300, initial_states=True, grad=True,
                                dfinal_states=True), False),
    # time-contiguous [B, D, T], rows of a multiple of 8 tokens
    ("dense_time_contiguous", dict(B=2, D=40, T=512, channel_last=False, initial_states=True,
                                   grad=True), False),
    # packed sequences, FP32 weight, no bias, deterministic
    ("packed", dict(B=1, D=512, T=325, lengths=[5, 120, 200], initial_states=True, grad=True,
                    bias=False, weight_dtype=torch.float32), True),
]


@pytest.mark.parametrize("name,kw,det", CASES, ids=[c[0] for c in CASES])
def test_graph_replay_matches_eager_and_oracle(name, kw, det, cuda_device):
    kw = dict(kw)
    B, D, T = kw.pop("B"), kw.pop("D"), kw.pop("T")
    inp = make_inputs(B, D, T, seed=5, deterministic=det, **kw)
    call = Call(inp, cuda_device, det)
    stream = torch.cuda.current_stream(cuda_device)
    call.launch(stream)
    torch.cuda.synchronize()
    assert call.read_status(stream) == _abi.CCC_OK
    eager = [t.clone() for t in call.outputs()]

    g = capture(call.launch, cuda_device)
    for _ in range(2):  # a second replay over poisoned outputs: nothing is left over
        for t in call.outputs():
            t.fill_(POISON)
        g.replay()
        torch.cuda.synchronize()
        assert call.read_status(stream) == _abi.CCC_OK
        for e, t in zip(eager, call.outputs()):
            assert torch.equal(e.view(torch.int16) if e.dtype == torch.bfloat16 else e,
                               t.view(torch.int16) if t.dtype == torch.bfloat16 else t)

    # the replayed results against the oracle
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(call.out.cpu()), ref["out"], "out")
    if call.fin is not None:
        assert_bits_equal(bits(call.fin.cpu()), ref["final"], "final_states")
    rb = oracle_bwd(inp)
    assert_bf16_close(bits(call.dx.cpu()), rb["dx"], "dx")
    assert_wgrad_close(tensor_values(call.dw), rb["dw64"], rb["dw_abs"],
                       inp.weight.dtype == torch.bfloat16, "dweight")
    if call.db is not None:
        assert_wgrad_close(tensor_values(call.db), rb["db64"], rb["db_abs"], True, "dbias")
    if call.dinit is not None:
        assert_bf16_close(bits(call.dinit.cpu()), rb["dinit"], "dinitial_states")


def test_graph_reports_offsets_rewritten_after_capture(cuda_device):
    """The offsets are device data read by the kernels: a graph captured over
    valid offsets, replayed after they are rewritten in place to a malformed
    array, records CCC_ERR_BAD_CU_SEQLENS; restored, it replays cleanly."""
    inp = make_inputs(1, 256, 90, seed=9, lengths=[30, 60], initial_states=True, grad=True,
                      bias=False, weight_dtype=torch.float32, deterministic=True)
    call = Call(inp, cuda_device, True)
    stream = torch.cuda.current_stream(cuda_device)
    good = call.d.cu_seqlens.clone()
    call.launch(stream)
    torch.cuda.synchronize()
    assert call.read_status(stream) == _abi.CCC_OK
    g = capture(call.launch, cuda_device)
    g.replay()
    torch.cuda.synchronize()
    assert call.read_status(stream) == _abi.CCC_OK
    call.d.cu_seqlens.copy_(torch.tensor([0, 60, 30], dtype=torch.int32))  # not increasing
    g.replay()
    torch.cuda.synchronize()
    assert call.read_status(stream) == _abi.CCC_ERR_BAD_CU_SEQLENS
    call.d.cu_seqlens.copy_(good)
    g.replay()
    torch.cuda.synchronize()
    assert call.read_status(stream) == _abi.CCC_OK
    ref = oracle_fwd(inp)
    assert_bf16_close(bits(call.out.cpu()), ref["out"], "out")


@pytest.mark.parametrize("B,D", [(8, 4096), (5, 100)])
def test_graph_update_chain(B, D, cuda_device):
    """Twelve chained single-token updates captured as one graph: bitwise the
    eager chain, and the oracle's forward over the twelve tokens with the
    starting state as initial state (its final state bitwise)."""
    steps = 12
    gen = torch.Generator().manual_seed(B + D)
    state0 = torch.randn(B, D, 3, generator=gen).to(torch.bfloat16)
    xs = torch.randn(steps, B, D, generator=gen).to(torch.bfloat16)
    w = (torch.rand(D, 4, generator=gen) - 0.5).to(torch.bfloat16)
    b = ((torch.rand(D, generator=gen) - 0.5) * 0.2).to(torch.bfloat16)
    dev = cuda_device
    xs_d, w_d, b_d = xs.to(dev), w.to(dev), b.to(dev)
    act = _abi.CCC_ACT_SILU
    stream = torch.cuda.current_stream(dev)

    s_e = state0.to(dev)
    out_e = torch.empty(steps, B, D, dtype=torch.bfloat16, device=dev)
    for i in range(steps):
        assert _abi.ccc_conv1d_update(xs_d[i], s_e, w_d, b_d, out_e[i], act, stream) == _abi.CCC_OK
    torch.cuda.synchronize()

    s_g = state0.to(dev)
    out_g = torch.empty(steps, B, D, dtype=torch.bfloat16, device=dev)

    def chain(s):
        for i in range(steps):
            assert _abi.ccc_conv1d_update(xs_d[i], s_g, w_d, b_d, out_g[i], act, s) == _abi.CCC_OK

    g = capture(chain, dev)
    s_g.copy_(state0.to(dev))  # capture records the launches without running them
    out_g.fill_(POISON)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(s_g.view(torch.int16), s_e.view(torch.int16))

    x_seq = xs.permute(1, 2, 0)  # [B, D, steps]: token i of row b is xs[i, b]
    ref = oracle.fwd(bits(x_seq), bits(w), bits(b), None, bits(state0), "silu")
    assert_bf16_close(bits(out_g.permute(1, 2, 0).cpu()), ref["out"], "out")
    assert_bits_equal(bits(s_g.cpu()), ref["final"], "state")
