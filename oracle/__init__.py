"""CPU oracle for the depthwise causal conv1d -- TEST INFRASTRUCTURE ONLY.

A plain, slow restatement of the operation (``conv1d_oracle.c``, fp64) behind a
numpy interface.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the library under
``depthwise_causal_conv1d_channel_gb300`` never does, and this package never
imports it.

Two layers:

* ``*_f64`` functions run the C core on float64 arrays of any real values (the
  finite-difference pins use these).
* ``fwd`` / ``bwd`` / ``update`` take BF16 inputs as ``np.uint16`` bit patterns
  (the weight may instead be float32), decode them exactly, run the core, and
  round each result once, nearest-even, to the output type: BF16 bits for
  activations, states and bias gradients; BF16 bits or float32 for the weight
  gradient, following the weight's dtype.  The float64 values are returned too.

Shapes: ``x`` / ``g`` are the logical ``[B, D, T]`` tensor (copied to
contiguous here); packed calls have ``B == 1`` and ``cu_seqlens`` of ``N + 1``
int32 offsets; ``weight`` is ``[D, W]`` with a width W in 2..4 (4 on the
page's optimized route); states are ``[B or N, D, W - 1]``.
What the core computes, and the page passages it follows, is written at the
top of ``conv1d_oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv1d_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

ACTIVATIONS = {"silu": 1, None: 0, "none": 0, "identity": 0}
BAD_CU_SEQLENS = 7
BAD_SEQ_IDX = 102

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C99, no FMA contraction, no fast-math)."""
    stale = not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-Wall", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        # CCC_ORACLE_LIB lets the oracle's own mutation tests load a deliberately
        # broken copy; nothing else sets it.
        lib = ctypes.CDLL(os.environ.get("CCC_ORACLE_LIB") or build())
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_fwd.argtypes = [P, I64, I64, I64, P, I, P, P, I, P, P, I, P, P, P]
        lib.oracle_fwd.restype = I
        lib.oracle_bwd.argtypes = [P, I64, I64, I64, P, I, P, P, I, P, P, I, P, P, P, P, P, P, P, P]
        lib.oracle_bwd.restype = I
        lib.oracle_update.argtypes = [P, I64, I64, P, I, P, I, P, P]
        lib.oracle_update.restype = I
        lib.oracle_check_cu_seqlens.argtypes = [P, I, I64]
        lib.oracle_check_cu_seqlens.restype = I
        lib.oracle_fullconv_fwd.argtypes = [P, I64, I64, I64, P, I64, I, I, P, P, P]
        lib.oracle_fullconv_fwd.restype = I
        lib.oracle_bf16_encode.argtypes = [ctypes.c_double]
        lib.oracle_bf16_encode.restype = ctypes.c_uint16
        lib.oracle_bf16_encode_array.argtypes = [P, I64, P]
        lib.oracle_bf16_encode_array.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _act(activation):
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation {activation!r} not supported")
    return ACTIVATIONS[activation]


def _seq_idx(x_shape, seq_idx):
    """Per-token sequence ids [B, T] as contiguous int32 (or None)."""
    if seq_idx is None:
        return None
    ids = np.ascontiguousarray(seq_idx, dtype=np.int32)
    if ids.shape != (x_shape[0], x_shape[2]):
        raise ValueError(f"seq_idx must be [B, T] = {(x_shape[0], x_shape[2])}, got {ids.shape}")
    return ids


def _cu(B, cu_seqlens):
    if cu_seqlens is None:
        return None, B
    if B != 1:
        raise ValueError("packed calls take batch 1")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    return cu, cu.shape[0] - 1


# ---- number formats ----------------------------------------------------------

def bf16_decode(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact)."""
    if bits is None:
        return None
    b = np.ascontiguousarray(bits)
    if b.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns (uint16), got {b.dtype}")
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_encode(v) -> np.ndarray:
    """float64 -> BF16 bit patterns, nearest-even (the oracle's own rounding)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def _weight_f64(weight):
    w = np.ascontiguousarray(weight)
    if w.dtype == np.uint16:
        return bf16_decode(w), False
    if w.dtype == np.float32:
        return w.astype(np.float64), True
    raise TypeError(f"weight must be BF16 bits (uint16) or float32, got {w.dtype}")


def _width(w) -> int:
    """The filter width W of a [D, W] weight (2..4)."""
    if w.ndim != 2 or not 2 <= w.shape[1] <= 4:
        raise ValueError(f"weight must be [D, W] with 2 <= W <= 4, got shape {w.shape}")
    return int(w.shape[1])


def check_cu_seqlens(cu_seqlens, total: int) -> bool:
    """True when the offsets follow the page's rules (first 0, last == total,
    strictly increasing)."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    return _load().oracle_check_cu_seqlens(_ptr(cu), cu.shape[0] - 1, int(total)) == 0


# ---- fp64 core ---------------------------------------------------------------

def _check_rc(rc, what):
    if rc == BAD_CU_SEQLENS:
        raise ValueError(f"malformed cu_seqlens (oracle status {rc})")
    if rc == BAD_SEQ_IDX:
        raise ValueError("seq_idx excludes cu_seqlens, initial states and final states")
    if rc != 0:
        raise ValueError(f"oracle {what} failed (status {rc})")


def fwd_f64(x, weight, bias=None, cu_seqlens=None, initial_states=None, activation="silu",
            seq_idx=None):
    """Returns dict(out, pre: [B,D,T], final: [S,D,W-1]) in float64 (final is None
    with seq_idx, which defines no state)."""
    lib = _load()
    x = _f64(x)
    B, D, T = x.shape
    w = _f64(weight)
    W = _width(w)
    cu, S = _cu(B, cu_seqlens)
    ids = _seq_idx(x.shape, seq_idx)
    out = np.empty((B, D, T))
    pre = np.empty((B, D, T))
    fin = np.empty((S, D, W - 1)) if ids is None else None
    rc = lib.oracle_fwd(_ptr(x), B, D, T, _ptr(w), W, _ptr(_f64(bias)), _ptr(cu), S, _ptr(ids),
                        _ptr(_f64(initial_states)), _act(activation), _ptr(out), _ptr(pre),
                        _ptr(fin))
    _check_rc(rc, "forward")
    return dict(out=out, pre=pre, final=fin)


def bwd_f64(x, weight, g, bias=None, cu_seqlens=None, initial_states=None, dfinal_states=None,
            activation="silu", seq_idx=None):
    """Returns dict(dx [B,D,T], dinit [S,D,W-1], dw, dw_abs [D,W], db, db_abs [D]) in
    float64.  ``dinit`` is the gradient at the W - 1 positions before each
    sequence, given whether or not initial states were passed."""
    lib = _load()
    x = _f64(x)
    B, D, T = x.shape
    w = _f64(weight)
    W = _width(w)
    g = _f64(g)
    if g.shape != x.shape:
        raise ValueError("g must have the shape of x")
    cu, S = _cu(B, cu_seqlens)
    ids = _seq_idx(x.shape, seq_idx)
    dx = np.empty((B, D, T))
    dinit = np.empty((S, D, W - 1))
    dw = np.empty((D, W))
    dw_abs = np.empty((D, W))
    db = np.empty((D,))
    db_abs = np.empty((D,))
    rc = lib.oracle_bwd(_ptr(x), B, D, T, _ptr(w), W, _ptr(_f64(bias)), _ptr(cu), S, _ptr(ids),
                        _ptr(_f64(initial_states)), _act(activation), _ptr(g),
                        _ptr(_f64(dfinal_states)), _ptr(dx), _ptr(dinit), _ptr(dw),
                        _ptr(dw_abs), _ptr(db), _ptr(db_abs))
    _check_rc(rc, "backward")
    return dict(dx=dx, dinit=dinit, dw=dw, dw_abs=dw_abs, db=db, db_abs=db_abs)


def update_f64(x, conv_state, weight, bias=None, activation="silu"):
    """Returns dict(out [B,D], state [B,D,W-1]) in float64; the input state is not modified."""
    lib = _load()
    x = _f64(x)
    B, D = x.shape
    w = _f64(weight)
    W = _width(w)
    state = np.array(conv_state, dtype=np.float64, copy=True)
    if state.shape != (B, D, W - 1):
        raise ValueError("conv_state must be [B, D, W - 1]")
    out = np.empty((B, D))
    lib.oracle_update(_ptr(x), B, D, _ptr(w), W, _ptr(_f64(bias)), _act(activation),
                      _ptr(state), _ptr(out))
    return dict(out=out, state=state)


# ---- BF16 interface ----------------------------------------------------------

def fwd(x, weight, bias=None, cu_seqlens=None, initial_states=None, activation="silu",
        seq_idx=None):
    """BF16 forward.  Returns dict(out, final: uint16 bits; out64, pre64, final64:
    float64); final and final64 are None with seq_idx."""
    w, _ = _weight_f64(weight)
    r = fwd_f64(bf16_decode(x), w, bf16_decode(bias), cu_seqlens, bf16_decode(initial_states),
                activation, seq_idx)
    fin = None if r["final"] is None else bf16_encode(r["final"])
    return dict(out=bf16_encode(r["out"]), out64=r["out"], pre64=r["pre"], final=fin,
                final64=r["final"])


def bwd(x, weight, g, bias=None, cu_seqlens=None, initial_states=None, dfinal_states=None,
        activation="silu", seq_idx=None):
    """BF16 backward.  Returns dict(dx, dinit, db: uint16 bits; dw: uint16 bits for a
    BF16 weight or float32 for an FP32 weight; dx64, dinit64, dw64, db64, dw_abs,
    db_abs: float64)."""
    w, w_f32 = _weight_f64(weight)
    r = bwd_f64(bf16_decode(x), w, bf16_decode(g), bf16_decode(bias), cu_seqlens,
                bf16_decode(initial_states), bf16_decode(dfinal_states), activation, seq_idx)
    dw = r["dw"].astype(np.float32) if w_f32 else bf16_encode(r["dw"])
    return dict(dx=bf16_encode(r["dx"]), dinit=bf16_encode(r["dinit"]), dw=dw,
                db=bf16_encode(r["db"]), dx64=r["dx"], dinit64=r["dinit"], dw64=r["dw"],
                db64=r["db"], dw_abs=r["dw_abs"], db_abs=r["db_abs"])


def update(x, conv_state, weight, bias=None, activation="silu"):
    """BF16 decode step.  Returns dict(out, state: uint16 bits; out64: float64)."""
    w, _ = _weight_f64(weight)
    r = update_f64(bf16_decode(x), bf16_decode(conv_state), w, bf16_decode(bias), activation)
    return dict(out=bf16_encode(r["out"]), out64=r["out"], state=bf16_encode(r["state"]))


# ---- full-channel dilated causal conv1d (POPCORNBENCH conv1d page) -----------

def fullconv_f64(x, weight, bias=None, dilation=1):
    """x [B, Cin, T], weight [Cout, Cin, K], bias [Cout] or None (any real values).
    Returns dict(out [B, Cout, T], abs_sum [B, Cout, T]) in float64."""
    lib = _load()
    x = _f64(x)
    w = _f64(weight)
    B, Cin, T = x.shape
    Cout, Cin_w, K = w.shape
    if Cin_w != Cin:
        raise ValueError("weight must be [Cout, Cin, K] with the Cin of x")
    out = np.empty((B, Cout, T))
    abs_sum = np.empty((B, Cout, T))
    rc = lib.oracle_fullconv_fwd(_ptr(x), B, Cin, T, _ptr(w), Cout, int(K), int(dilation),
                                 _ptr(_f64(bias)), _ptr(out), _ptr(abs_sum))
    if rc != 0:
        raise ValueError(f"kernel size and dilation must be >= 1 (oracle status {rc})")
    return dict(out=out, abs_sum=abs_sum)


def fullconv(x, weight, bias=None, dilation=1):
    """BF16 inputs (uint16 bit patterns; weight and bias may be float32 instead).
    Returns dict(out: BF16 bits, out64, abs_sum: float64)."""
    w = bf16_decode(weight) if np.asarray(weight).dtype == np.uint16 else _f64(weight)
    b = None if bias is None else (bf16_decode(bias) if np.asarray(bias).dtype == np.uint16
                                   else _f64(bias))
    r = fullconv_f64(bf16_decode(x), w, b, dilation)
    return dict(out=bf16_encode(r["out"]), out64=r["out"], abs_sum=r["abs_sum"])
