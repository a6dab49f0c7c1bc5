"""Throughput of the depthwise causal conv1d on GB300: forward + backward of the
large dense channel-last workload (x stored [8, 8192, 5120] BF16, BF16
weight/bias, initial/final state, grad_out) -- the largest of the workloads,
all of which fit one GPU -- as achieved HBM GB/s (algorithmic bytes / time)
and tokens/s, with the other workloads (dense [2, 64, 128] forward, dense
[4, 2048, 1536] with state, packed varlen, decode update, the large dense
workload bias-free and deterministic) reported per kernel under "breakdown".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Under torchrun (N > 1) every rank runs the same
workload on its own GPU (independent replicas, no collective on the data
path); the time is the max over ranks and the value counts all ranks' work.

--impl reference times the CPU oracle (oracle/, plain C in fp64) on the host
cores on a bounded sample of the same workload: the only comparison system the
pages leave us, a deliberately slow baseline.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fwd/bwd/update achieved HBM GB/s and tokens/s vs ~8 TB/s GB300 peak"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant
# call -- the backward on the large dense workload: backward kernel plus the
# finalize kernel -- from one ncu capture of those two kernels
# (profiles/traffic_dense_large_backward.md), per launch.  Valid only for the
# kernel sources whose digest (of their code, comments left out) is recorded
# here (null otherwise).
TRAFFIC = {"sources_sha256": "ca39b3737eccc7cde07475d8cdaed24dde08245357eb9d70255bb78de46dad71",
           "bytes_per_launch": (1349984256 + 634317056) + (1543168 + 0)}


# The sources the dominant call's kernels (the channel-last backward and the
# finalize) and their launch plan are built from.
TRAFFIC_SOURCES = ("abi.cu", "bwd.cu", "common.cuh", "launch.h")


def _code_only(text: str) -> str:
    """The source without its comments and blank lines (an edited comment
    leaves the recorded traffic valid; any change to the code does not)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_sources_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "depthwise_causal_conv1d_channel_gb300", "csrc")
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()


def recorded_traffic():
    """DRAM bytes per launch of the dominant call, or None once the code it was
    captured from has changed."""
    return TRAFFIC["bytes_per_launch"] if TRAFFIC["sources_sha256"] == kernel_sources_digest() else None


# ---- sizes ------------------------------------------------------------------------

def act_bytes(x):
    return x.numel() * x.element_size()


def fwd_bytes(x, w, b, init, fin):
    """Algorithmic minimum: read x, write out, read weight/bias/initial state,
    write final state."""
    n = 2 * act_bytes(x) + act_bytes(w)
    for t in (b, init, fin):
        if t is not None:
            n += act_bytes(t)
    return n


def bwd_bytes(x, w, b, init, dfin, dinit):
    """Read x and grad_out, write dx, read weight, write dweight, read bias and
    write dbias, read initial state / final-state gradient, write dinitial_states."""
    n = 3 * act_bytes(x) + 2 * act_bytes(w)
    if b is not None:
        n += 2 * act_bytes(b)
    for t in (init, dfin, dinit):
        if t is not None:
            n += act_bytes(t)
    return n


def update_bytes(B, D, w, b):
    """Read and write the [B, D, 3] state, read x, write out, read weight/bias."""
    n = 2 * B * D * 3 * 2 + 2 * B * D * 2 + act_bytes(w)
    if b is not None:
        n += act_bytes(b)
    return n


# ---- clocks -----------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    p = [s.strip() for s in line.split(",")]
                    if len(p) >= 9 and p[1].isdigit():
                        rows.append(p)
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


def measured_peak(key="hbm_gbs", fallback=FALLBACK_HBM_GBS):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)[key])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return fallback, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


# ---- the timed step ---------------------------------------------------------------

class DenseStep:
    """Forward + backward through the C ABI on preallocated device buffers.
    `sets` copies of the activations rotate so that no step finds its inputs
    in L2 (total footprint well above the L2 size)."""

    def __init__(self, inp: workloads.ConvInputs, device, deterministic=False, sets=None,
                 seq_idx=None):
        from depthwise_causal_conv1d_channel_gb300 import _abi

        self.abi = _abi
        self.dev = device
        d = inp.to(device)
        self.inp = inp
        self.w, self.b, self.cu = d.weight, d.bias, d.cu_seqlens
        self.init, self.dfin = d.initial_states, d.dfinal_states
        self.det = deterministic
        self.act = _abi.CCC_ACT_SILU if inp.activation == "silu" else _abi.CCC_ACT_NONE
        per_set = 4 * act_bytes(d.x)
        if sets is None:
            sets = max(1, min(16, -(-3 * L2_BYTES // per_set)))
        self.sets = sets
        self.x = [d.x if i == 0 else d.x.clone() if not inp.channel_last else
                  d.x.transpose(1, 2).clone().transpose(1, 2) for i in range(sets)]
        self.g = [None if d.g is None else d.g if i == 0 else
                  d.g.transpose(1, 2).clone().transpose(1, 2) if inp.channel_last else
                  d.g.clone() for i in range(sets)]
        self.out = [torch.empty_like(x) for x in self.x]
        self.dx = [torch.empty_like(x) for x in self.x]
        S = inp.n_seq
        D = d.x.shape[1]
        W = d.weight.shape[1]
        self.fin = (torch.empty(S, D, W - 1, dtype=torch.bfloat16, device=device)
                    if self.init is not None else None)
        self.dinit = torch.empty_like(self.init) if self.init is not None else None
        self.dw = torch.empty_like(self.w)
        self.db = torch.empty_like(self.b) if self.b is not None else None
        self.ws = torch.empty(_abi.ccc_conv1d_bwd_workspace_size(d.x, deterministic),
                              dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ids = None if seq_idx is None else seq_idx.to(device)
        ids_bytes = 0 if seq_idx is None else act_bytes(seq_idx)
        self.fwd_bytes = fwd_bytes(d.x, self.w, self.b, self.init, self.fin) + ids_bytes
        self.bwd_bytes = bwd_bytes(d.x, self.w, self.b, self.init, self.dfin, self.dinit) + ids_bytes
        self.tokens = inp.tokens if inp.cu_seqlens is None else d.x.shape[2]
        self.launches_fwd = 1
        # backward kernel + the fixed-order finalize kernel
        self.launches_bwd = 2

    def fwd(self, i, stream):
        k = i % self.sets
        rc = self.abi.ccc_conv1d_fwd(self.x[k], self.w, self.b, self.cu, self.init, self.out[k],
                                     self.fin, self.act, self.status, stream, seq_idx=self.ids)
        assert rc == 0, self.abi.status_string(rc)

    def bwd(self, i, stream):
        k = i % self.sets
        rc = self.abi.ccc_conv1d_bwd(self.x[k], self.w, self.b, self.cu, self.init, self.g[k],
                                     self.dfin, self.dx[k], self.dw, self.db, self.dinit, self.act,
                                     self.det, self.ws, self.status, stream, seq_idx=self.ids)
        assert rc == 0, self.abi.status_string(rc)

    def check_status(self, stream):
        rc = self.abi.ccc_read_status(self.status, stream)
        assert rc == 0, self.abi.status_string(rc)


def _graph_of(fn, device, eager_first=True):
    """Capture fn(stream) into a CUDA graph (after one eager call, by default)."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        if eager_first:
            fn(torch.cuda.current_stream(device))
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn(torch.cuda.current_stream(device))
    torch.cuda.synchronize()
    return g


def time_fwd_bwd(step: DenseStep, steps: int, warmup: int, stream, barrier=lambda: None):
    """W eager warm-up steps; then the K steps as two CUDA graphs -- the K
    forward calls (buffer set k % sets for step k), then the K backward calls,
    as a training step runs every forward before every backward -- each
    replayed once untimed (graph upload) and then once timed, with events on
    the launching stream before, between and after the two replays.  Returns
    the total and the per-call forward and backward times."""
    n = step.sets
    for i in range(warmup):
        step.fwd(i % n, stream)
        step.bwd(i % n, stream)
    torch.cuda.synchronize()
    dev = step.dev
    fg = _graph_of(lambda s: [step.fwd((warmup + i) % n, s) for i in range(steps)], dev,
                   eager_first=False)
    bg = _graph_of(lambda s: [step.bwd((warmup + i) % n, s) for i in range(steps)], dev,
                   eager_first=False)
    fg.replay()
    bg.replay()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    barrier()
    torch.cuda.synchronize()
    ev[0].record(stream)
    fg.replay()
    ev[1].record(stream)
    bg.replay()
    ev[2].record(stream)
    torch.cuda.synchronize()
    barrier()
    step.check_status(stream)
    fwd_ms = ev[0].elapsed_time(ev[1]) / steps
    bwd_ms = ev[1].elapsed_time(ev[2]) / steps
    return ev[0].elapsed_time(ev[2]), fwd_ms, bwd_ms


# ---- breakdown over the other workloads ---------------------------------------------

def _per_call_ms(call, sets, device, stream, per=20, reps=5):
    """Median over `reps` replays of one graph holding `per` calls on rotating
    buffer sets: per-call device time with launch overhead amortised."""
    g = _graph_of(lambda s: [call(i % sets, s) for i in range(per)], device)
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / per)
    return statistics.median(out)


def bench_conv_workload(name, inp, device, stream, peak, deterministic, do_bwd=True, seq_idx=None):
    st = DenseStep(inp, device, deterministic=deterministic, seq_idx=seq_idx)
    r = {"workload": name, "tokens": st.tokens, "rotating_sets": st.sets}
    f_ms = _per_call_ms(st.fwd, st.sets, device, stream)
    r["fwd"] = _rate(st.fwd_bytes, f_ms, st.tokens, peak)
    if do_bwd:
        b_ms = _per_call_ms(st.bwd, st.sets, device, stream)
        r["bwd"] = _rate(st.bwd_bytes, b_ms, st.tokens, peak)
    st.check_status(stream)
    del st
    torch.cuda.empty_cache()
    return r


def _rate(nbytes, ms, tokens, peak):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"us": round(ms * 1e3, 2), "bytes": int(nbytes), "GB/s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "tokens_per_s": round(tokens / (ms * 1e-3))}


def bench_stream_floor(inp: workloads.ConvInputs, device, stream, peak):
    """Context for the dense workloads, not a roofline: PyTorch's own
    elementwise kernels moving the bytes of the dense forward (read x, write
    out: neg) and backward (read x and grad_out, write dx: add) on contiguous
    BF16 tensors of x's size, timed like the conv calls (a graph of 20 calls
    over rotating buffer sets, cold in L2)."""
    n = inp.x.numel()
    nbytes = 2 * n
    sets = max(1, -(-3 * L2_BYTES // (3 * nbytes)))
    gen = torch.Generator(device=device).manual_seed(0)
    a = [torch.randn(n, device=device, generator=gen).to(torch.bfloat16) for _ in range(sets)]
    b = [torch.randn(n, device=device, generator=gen).to(torch.bfloat16) for _ in range(sets)]
    o = [torch.empty_like(t) for t in a]
    neg_ms = _per_call_ms(lambda i, s: torch.neg(a[i % sets], out=o[i % sets]), sets, device, stream)
    add_ms = _per_call_ms(lambda i, s: torch.add(a[i % sets], b[i % sets], out=o[i % sets]), sets,
                          device, stream)
    return {"workload": "torch_elementwise_same_bytes", "elements": n, "rotating_sets": sets,
            "neg_1read_1write": _rate(2 * nbytes, neg_ms, inp.tokens, peak),
            "add_2read_1write": _rate(3 * nbytes, add_ms, inp.tokens, peak)}


def bench_update(device, stream, peak, iters=50, busy_s=0.0):
    from depthwise_causal_conv1d_channel_gb300 import _abi

    gen = torch.Generator(device=device).manual_seed(0)
    B, D = 256, 4096
    per = B * D * 3 * 2 + 2 * B * D * 2
    sets = max(1, -(-3 * L2_BYTES // per))
    state = [torch.randn(B, D, 3, device=device, generator=gen).to(torch.bfloat16) for _ in range(sets)]
    x = [torch.randn(B, D, device=device, generator=gen).to(torch.bfloat16) for _ in range(sets)]
    out = [torch.empty(B, D, dtype=torch.bfloat16, device=device) for _ in range(sets)]
    w = (torch.rand(D, 4, device=device, generator=gen) - 0.5).to(torch.bfloat16)
    b = ((torch.rand(D, device=device, generator=gen) - 0.5) * 0.2).to(torch.bfloat16)

    def upd(i, s):
        k = i % sets
        rc = _abi.ccc_conv1d_update(x[k], state[k], w, b, out[k], _abi.CCC_ACT_SILU, s)
        assert rc == 0

    ms = _per_call_ms(upd, sets, device, stream, per=40)
    r = {"workload": "decode_update", "batch": B, "dim": D, "rotating_sets": sets,
         "update": _rate(update_bytes(B, D, w, b), ms, B, peak)}
    # 1000 chained steps on one state in one CUDA graph (hot in L2; context only)
    g = _graph_of(lambda s: [upd(0, s) for _ in range(1000)], device)
    torch.cuda.synchronize()
    a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    c.record(stream)
    torch.cuda.synchronize()
    r["graph_chain_1000"] = {"us_per_step": round(a.elapsed_time(c) * 1e3 / 1000, 3),
                             "note": "one state, L2-resident, CUDA graph; not an HBM figure"}
    t_end = time.time() + busy_s  # untimed replays, so that clock samples see the load
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    return r


def bench_update_clocked(device, stream, peak, gpu_index):
    """bench_update with the SM clock sampled meanwhile: the step time times the
    median SM clock (thousands of cycles a step) separates the clock from the
    step's latency."""
    with ClockSampler(gpu_index) as clk:
        r = bench_update(device, stream, peak, busy_s=1.5)
    c = clk.summary()
    r["clocks"] = c
    if c.get("sm_mhz"):
        u = r["update"]
        u["kcycles_per_step"] = round(u["us"] * c["sm_mhz"] / 1000.0, 2)
        r["graph_chain_1000"]["kcycles_per_step"] = round(
            r["graph_chain_1000"]["us_per_step"] * c["sm_mhz"] / 1000.0, 2)
    return r


def bench_update_multi(device, stream, peak, L=4):
    """The update with L new tokens a row ([B, D, L], the multi-token form):
    B 256, D 4096, as the decode workload.  Bytes: state read and write, L
    tokens of x read and of out written, weight and bias."""
    from depthwise_causal_conv1d_channel_gb300 import _abi

    gen = torch.Generator(device=device).manual_seed(1)
    B, D = 256, 4096
    per = B * D * 3 * 2 + 2 * B * D * L * 2
    sets = max(1, -(-3 * L2_BYTES // per))
    state = [torch.randn(B, D, 3, device=device, generator=gen).to(torch.bfloat16) for _ in range(sets)]
    x = [torch.randn(B, L, D, device=device, generator=gen).to(torch.bfloat16).transpose(1, 2)
         for _ in range(sets)]
    out = [torch.empty(B, L, D, dtype=torch.bfloat16, device=device).transpose(1, 2)
           for _ in range(sets)]
    w = (torch.rand(D, 4, device=device, generator=gen) - 0.5).to(torch.bfloat16)
    b = ((torch.rand(D, device=device, generator=gen) - 0.5) * 0.2).to(torch.bfloat16)

    def upd(i, s):
        k = i % sets
        rc = _abi.ccc_conv1d_update(x[k], state[k], w, b, out[k], _abi.CCC_ACT_SILU, s)
        assert rc == 0

    ms = _per_call_ms(upd, sets, device, stream, per=40)
    nbytes = update_bytes(B, D, w, b) + 2 * B * D * (L - 1) * 2
    return {"workload": "decode_update_multi_token", "batch": B, "dim": D, "tokens_per_row": L,
            "rotating_sets": sets, "update": _rate(nbytes, ms, B * L, peak)}


def fullconv_flops(B, T, Cin, Cout, K):
    """Dense count of the full-channel conv: 2 * Cin * K multiply-adds per output
    (the taps that read the causal padding included)."""
    return 2 * B * T * Cout * Cin * K


class FullConvStep:
    """The full-channel dilated conv forward through the C ABI on the packed
    weight (packed once, outside the timed region)."""

    def __init__(self, inp: "workloads.FullConvInputs", device, sets=2):
        from depthwise_causal_conv1d_channel_gb300 import _abi
        import depthwise_causal_conv1d_channel_gb300 as ccc

        self.abi = _abi
        d = inp.to(device)
        self.dil = inp.dilation
        self.B, self.Cin, self.T = d.x.shape
        self.Cout, _, self.K = d.weight.shape
        self.packed = ccc.pack_full_conv_weight(d.weight)
        self.bias = d.bias
        self.sets = sets
        self.x = [d.x] + [d.x.transpose(1, 2).clone().transpose(1, 2) for _ in range(sets - 1)]
        self.out = [torch.empty(self.B, self.T, self.Cout, dtype=torch.bfloat16,
                                device=device).transpose(1, 2) for _ in range(sets)]
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.flops = fullconv_flops(self.B, self.T, self.Cin, self.Cout, self.K)

    def fwd(self, i, stream):
        k = i % self.sets
        rc = self.abi.ccc_fullconv1d_fwd(self.x[k], self.packed, self.bias, self.dil, self.out[k],
                                         self.status, stream)
        assert rc == 0, self.abi.status_string(rc)

    def check_status(self, stream):
        rc = self.abi.ccc_read_status(self.status, stream)
        assert rc == 0, self.abi.status_string(rc)


def bench_fullconv(device, stream):
    """The full-channel dilated causal conv (8 x 4096 tokens, 1024 -> 1024
    channels, K 4, dilation 2): TFLOP/s against the measured dense BF16 peak."""
    peak, kind = measured_peak("bf16_tflops", FALLBACK_BF16_TFLOPS)
    sustained, _ = measured_peak("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS)
    st = FullConvStep(workloads.fullconv_dilated(), device)
    ms = _per_call_ms(st.fwd, st.sets, device, stream)
    st.check_status(stream)
    tflops = st.flops / (ms * 1e-3) / 1e12
    r = {"workload": "fullconv_dilated", "B": st.B, "T": st.T, "Cin": st.Cin, "Cout": st.Cout,
         "K": st.K, "dilation": st.dil,
         "fwd": {"us": round(ms * 1e3, 2), "flops": st.flops, "TFLOP/s": round(tflops, 1),
                 "tokens_per_s": round(st.B * st.T / (ms * 1e-3))},
         "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                      "peak_kind": f"{kind} bf16 burst", "unit": "TFLOP/s",
                      "frac": round(tflops / peak, 4),
                      "frac_of_sustained": round(tflops / sustained, 4)}}
    del st
    torch.cuda.empty_cache()
    return r


# ---- end to end through the public API with host buffers ----------------------------

def time_e2e(inp: workloads.ConvInputs, device, steps, warmup, stream):
    """causal_conv1d + autograd backward, with each step's inputs copied from
    pinned host memory and every result copied back, inside the timed region.
    Inputs go up on their own stream into two device buffer sets, the way a
    training loop feeds a GPU, and results come down on a third: step i+1's
    inputs upload while step i's results download and step i+1 computes, so
    both directions of the host link stay busy (the link is the bound: about
    170 GB/s each way when both run, measured on the GB300's host link)."""
    import depthwise_causal_conv1d_channel_gb300 as ccc

    def pinned(t):
        if t is None:
            return None
        if inp.channel_last and t.dim() == 3 and t.shape == inp.x.shape:
            return t.transpose(1, 2).contiguous().pin_memory()  # [B, T, D] storage
        return t.contiguous().pin_memory()

    hx, hg = pinned(inp.x), pinned(inp.g)
    hw, hb, hi = pinned(inp.weight), pinned(inp.bias), pinned(inp.initial_states)
    S, D = inp.n_seq, inp.x.shape[1]
    ho = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    hf = torch.empty(S, D, inp.weight.shape[1] - 1, dtype=torch.bfloat16).pin_memory()
    hdi = torch.empty_like(hi).pin_memory()
    hdw = torch.empty_like(hw).pin_memory()
    hdb = torch.empty_like(hb).pin_memory() if hb is not None else None
    h_in = [t for t in (hx, hg, hw, hb, hi) if t is not None]
    h2d = sum(act_bytes(t) for t in h_in)
    d2h = sum(act_bytes(t) for t in (ho, hdx, hf, hdi, hdw, hdb) if t is not None)

    comp = stream
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    dev = [[torch.empty_like(t, device=device) for t in h_in] for _ in range(2)]
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def upload(j, after):
        if after is not None:
            s_in.wait_event(after)
        with torch.cuda.stream(s_in):
            for d, h in zip(dev[j], h_in):
                d.copy_(h, non_blocking=True)
        in_done[j].record(s_in)

    def compute(j):
        comp.wait_event(in_done[j])
        x, g, w, b, init = (t.detach() for t in dev[j])
        if inp.channel_last:
            x, g = x.transpose(1, 2), g.transpose(1, 2)
        for t in (x, w, b, init):
            t.requires_grad_(True)
        out, fin = ccc.causal_conv1d(x, w, b, initial_states=init, return_final_states=True)
        out.backward(g)
        comp_done[j].record(comp)  # the kernels are done with buffer set j
        res = [out.detach().transpose(1, 2) if inp.channel_last else out.detach(),
               x.grad.transpose(1, 2) if inp.channel_last else x.grad,
               fin.detach(), init.grad, w.grad, b.grad]
        s_out.wait_event(comp_done[j])
        with torch.cuda.stream(s_out):
            for h, r in zip((ho, hdx, hf, hdi, hdw, hdb), res):
                if r is not None:
                    h.copy_(r, non_blocking=True)
                    r.record_stream(s_out)  # not reused before its download ends

    def run(n):
        upload(0, None)
        for i in range(n):
            if i + 1 < n:  # buffer set (i+1) % 2 was last read by step i-1
                upload((i + 1) % 2, comp_done[(i + 1) % 2] if i >= 1 else None)
            compute(i % 2)

    run(max(warmup, 2))
    torch.cuda.synchronize()
    # three timed passes of `steps` steps each; the median pass is reported (the
    # host link's rate varies a little from pass to pass)
    times = []
    for _ in range(3):
        a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        run(steps)
        comp.wait_stream(s_out)
        comp.wait_stream(s_in)
        c.record(comp)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(c) / steps)
    return statistics.median(times), h2d, d2h


# ---- CPU oracle ---------------------------------------------------------------------

def host_cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (best effort)."""
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ":" in ln:
                    k, v = ln.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        for k in ("model name", "Model", "CPU part"):
            if k in fields:
                impl = fields.get("CPU implementer", "")
                return fields[k] if k != "CPU part" else f"implementer {impl} part {fields[k]}"
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_threads() -> int:
    """Host cores this process may run on (the oracle is split over them)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_step_seconds(inp, min_seconds=10.0, max_reps=20, channels=None, threads=1):
    """The oracle's forward + backward on the workload (all channels unless a
    sample is given), repeated until `min_seconds` have passed.  Channels are
    independent, so the channel list is split into `threads` contiguous chunks
    run at once on a thread pool (the oracle's C calls release the GIL); each
    chunk's inputs are sliced and converted before the clock starts."""
    import concurrent.futures
    import numpy as np

    import oracle
    from workloads import bits

    D = inp.x.shape[1]
    chans = list(range(D)) if channels is None else list(channels)
    threads = max(1, min(threads, len(chans)))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    jobs = []
    for chunk in np.array_split(np.array(chans), threads):
        c = chunk.tolist()
        b = inp.bias[c] if inp.bias is not None else None
        init = inp.initial_states[:, c] if inp.initial_states is not None else None
        jobs.append((bits(inp.x[:, c]), bits(inp.weight[c]), bits(b), bits(init), bits(inp.g[:, c])))

    def run(job):
        x, w, b, init, g = job
        oracle.fwd(x, w, b, cu, init, inp.activation)
        oracle.bwd(x, w, g, b, cu, init, None, inp.activation)

    reps = 0
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        while True:
            list(pool.map(run, jobs))
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or reps >= max_reps:
                break
    x = inp.x[:, chans]
    w = inp.weight[chans]
    b = inp.bias[chans] if inp.bias is not None else None
    init = inp.initial_states[:, chans] if inp.initial_states is not None else None
    nb = fwd_bytes(x, w, b, init, init) + bwd_bytes(x, w, b, init, None, init)
    return el / reps, nb, reps, x.shape


# ---- main ---------------------------------------------------------------------------

def reduce_max(value: float, device) -> float:
    """Max of a per-rank number over all ranks (the job's time is the slowest
    rank's)."""
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def headline_config(world: int) -> dict:
    """The timed workload, shared by both arms: forward + backward of the large
    dense workload (BF16 x stored [8, 8192, 5120], seen as [8, 5120, 8192])."""
    B, D, T = 8, 5120, 8192
    act_mb = B * T * D * 2 / 1e6
    return {"workload": "dense_large", "x": [B, D, T],
            "layout": f"channel-last ([{B}, {T}, {D}] storage)",
            "weight": "bf16", "bias": True, "initial_states": True,
            "final_states": True, "dweight": "fp32-partials",
            "step": "forward + backward", "parallelism": f"replicas{world}",
            "l2": f"inputs larger than L2: x and grad_out {act_mb:.0f} MB each, one buffer set"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = workloads.dense_large(bias=True)
    D = inp.x.shape[1]
    channels = list(range(0, D, 64))  # a 1/64 sample of the channels, every token
    threads = oracle_threads()
    ms = []
    for _ in range(args.warmup):
        oracle_step_seconds(inp, 0.0, 1, channels, threads)
    for _ in range(args.steps):
        s, nb, reps, shape = oracle_step_seconds(inp, 0.0, 1, channels, threads)
        ms.append(s * 1e3)
    per = statistics.mean(ms)
    value = nb / (per * 1e-3) / 1e9
    sample = (f"dense_large workload, forward+backward on {len(channels)} of {D} channels "
              f"(every 64th), all {inp.tokens} tokens, per step, split over {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PROFILE_WORKLOADS = ("dense_small", "dense_state", "dense_state_time_contiguous", "packed_varlen",
                     "decode_update", "dense_large_bias", "dense_large_det",
                     "dense_large_quarter", "fullconv_dilated")


def run_profile(name: str, calls: int):
    """A few eager calls of one workload's kernels and nothing else, for an ncu
    launch list or capture: forward + backward (or the update)."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from depthwise_causal_conv1d_channel_gb300 import _abi

    stream = torch.cuda.current_stream(device)
    if name == "fullconv_dilated":
        st = FullConvStep(workloads.fullconv_dilated(), device, sets=1)
        for _ in range(calls):
            st.fwd(0, stream)
        st.check_status(stream)
        torch.cuda.synchronize()
        print(json.dumps({"profile": name, "calls": calls}))
        return
    if name == "decode_update":
        wl = workloads.decode_update(steps=calls)
        st = wl.conv_state.to(device)
        w, b = wl.weight.to(device), wl.bias.to(device)
        out = torch.empty(st.shape[0], st.shape[1], dtype=torch.bfloat16, device=device)
        for i in range(calls):
            assert _abi.ccc_conv1d_update(wl.x_seq[i].to(device), st, w, b, out,
                                          _abi.CCC_ACT_SILU, stream) == 0
    else:
        if name == "dense_small":
            inp = workloads.dense_small()
        elif name == "dense_state":
            inp = workloads.dense_state()
        elif name == "dense_state_time_contiguous":
            inp = workloads.make_inputs(4, 1536, 2048, seed=0, initial_states=True, grad=True,
                                        channel_last=False)
        elif name == "packed_varlen":
            inp = workloads.packed_varlen()
        elif name == "dense_large_quarter":
            # the large workload's shape with a quarter of its tokens (x and
            # grad_out 168 MB each, still above L2): the small case for
            # multi-pass ncu captures of its kernels
            inp = workloads.make_inputs(8, 5120, 2048, seed=0, initial_states=True, grad=True)
        else:
            inp = workloads.dense_large(bias=name == "dense_large_bias")
        step = DenseStep(inp, device, deterministic=inp.deterministic, sets=1)
        for i in range(calls):
            step.fwd(0, stream)
            if step.g[0] is not None:
                step.bwd(0, stream)
        step.check_status(stream)
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "calls": calls}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=PROFILE_WORKLOADS,
                    help="run only a few eager calls of this workload (for ncu) and exit")
    ap.add_argument("--calls", type=int, default=3)
    args = ap.parse_args()
    if args.profile:
        return run_profile(args.profile, args.calls)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        pg = dist
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import depthwise_causal_conv1d_channel_gb300  # noqa: F401  (loads the CUDA library)

    stream = torch.cuda.current_stream(device)
    peak, peak_kind = measured_peak()
    # the largest workload: x and grad_out are 671 MB each, larger than L2, so
    # one buffer set serves every step cold
    inp = workloads.dense_large(bias=True)
    step = DenseStep(inp, device, sets=1)

    def barrier():
        if pg is not None:
            pg.barrier()

    with ClockSampler(local) as clk:
        total_ms, f_ms, b_ms = time_fwd_bwd(step, args.steps, args.warmup, stream, barrier)
    clocks = clk.summary()

    ms_step = total_ms / args.steps
    if pg is not None:
        ms_step = reduce_max(ms_step, device)
    step_bytes = step.fwd_bytes + step.bwd_bytes
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    tokens_per_s = world * step.tokens / (ms_step * 1e-3)

    dominant = ("bwd", b_ms, step.bwd_bytes) if b_ms >= f_ms else ("fwd", f_ms, step.fwd_bytes)
    achieved = dominant[2] / (dominant[1] * 1e-3) / 1e9
    traffic = recorded_traffic()

    e2e_ms, h2d, d2h = time_e2e(inp, device, args.steps, args.warmup, stream)
    e2e_value = world * step_bytes / (e2e_ms * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(world),
        "tokens_per_s": round(tokens_per_s),
        "fwd_us": round(f_ms * 1e3, 2), "bwd_us": round(b_ms * 1e3, 2),
        "gpu_launches": args.steps * (step.launches_fwd + step.launches_bwd),
        "timing": "K forward calls then K backward calls, each as one CUDA graph replay "
                  "(after an untimed upload replay); events before, between and after",
        "roofline": {"bound": "hbm", "kernel": f"{dominant[0]} call (dense_large)",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "bytes_per_launch": dominant[2]},
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "api": "causal_conv1d + autograd backward",
                "copies": "pinned host buffers; uploads and downloads each on their own "
                          "stream (two device input sets), overlapping each other and the "
                          "compute of the step between them (each step's copies inside the "
                          "timed region); median of three timed passes of --steps steps"},
    }

    if not args.no_breakdown:
        del step
        torch.cuda.empty_cache()
        ds = workloads.dense_state()
        bd = [bench_conv_workload("dense_small", workloads.dense_small(), device, stream, peak,
                                  False, do_bwd=False),
              bench_conv_workload("dense_state", ds, device, stream, peak, False),
              bench_stream_floor(ds, device, stream, peak),
              bench_conv_workload("packed_varlen", workloads.packed_varlen(), device, stream, peak,
                                  True),
              bench_update_clocked(device, stream, peak, local)]
        # the same dense step on a contiguous [B, D, T] tensor (time-contiguous)
        tc = workloads.make_inputs(4, 1536, 2048, seed=0, initial_states=True, grad=True,
                                   channel_last=False)
        bd.append(bench_conv_workload("dense_state_time_contiguous", tc, device, stream, peak, False))
        # the same dense step with a width-three filter (weight [D, 3], states [., D, 2])
        w3 = workloads.make_inputs(4, 1536, 2048, seed=0, initial_states=True, grad=True, width=3)
        bd.append(bench_conv_workload("dense_state_width3", w3, device, stream, peak, False))
        # the dense_state shape (no states) with per-token sequence ids: runs of
        # U[1, 512] tokens in every row
        si = workloads.make_inputs(4, 1536, 2048, seed=0, grad=True)
        bd.append(bench_conv_workload("dense_state_seq_idx", si, device, stream, peak, False,
                                      seq_idx=workloads.seq_ids(4, 2048, seed=0, max_run=512)))
        bd.append(bench_update_multi(device, stream, peak))
        bd.append(bench_conv_workload("dense_large_bias", inp, device, stream, peak, False))
        large = dataclasses.replace(inp, bias=None, deterministic=True)
        bd.append(bench_conv_workload("dense_large_det", large, device, stream, peak, True))
        bd.append(bench_fullconv(device, stream))
        line["breakdown"] = bd

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = oracle_threads()
        D = inp.x.shape[1]
        chans = list(range(0, D, 32))  # every 32nd channel, all tokens
        s, nb, reps, shape = oracle_step_seconds(inp, 1.5, 200, chans, threads)
        s1, nb1, reps1, _ = oracle_step_seconds(inp, 1.0, 5, chans[:len(chans) // 8], 1)
        line["cpu_baseline"] = {"value": round(nb / s / 1e9, 4), "unit": UNIT, "cores": threads,
                                "kind": "oracle", "cpu": host_cpu_model(),
                                "sample": f"dense_large workload fwd+bwd on {len(chans)} of {D} "
                                          f"channels (every 32nd), all {inp.tokens} tokens; "
                                          f"channels split over {threads} threads, {reps} reps, "
                                          f"{s:.3f} s each ({reps * s * threads:.0f} core-seconds)",
                                "single_thread": {"value": round(nb1 / s1 / 1e9, 4), "cores": 1,
                                                  "sample": f"{len(chans) // 8} of those channels, "
                                                            f"one thread, {reps1} reps, "
                                                            f"{s1:.2f} s each"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
