"""CPU-only checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments on the host before touching any
device memory.  The data pointers below are never dereferenced: every call here
fails a host-side check that runs before the first CUDA call.
"""

import ctypes
import os
import re

import pytest

from conftest import ROOT

import depthwise_causal_conv1d_channel_gb300 as ccc
from depthwise_causal_conv1d_channel_gb300 import _abi

HEADER = os.path.join(ROOT, "include", "ccc_conv1d.h")

BF16, F32, I32 = _abi.CCC_BF16, _abi.CCC_F32, _abi.CCC_I32


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ccc_\w+)\s*\(", src)))


def test_header_declarations_are_exported():
    names = declared_functions()
    assert set(names) == set(_abi.EXPORTED)
    lib = ctypes.CDLL(ccc._abi.lib._name)
    for n in names:
        assert hasattr(lib, n), n


def test_header_compiles_as_c():
    import subprocess
    import tempfile

    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        with open(src, "w") as f:
            f.write('#include "ccc_conv1d.h"\nint main(void){return ccc_conv1d_abi_version() != '
                    'CCC_CONV1D_ABI_VERSION;}\n')
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", src, "-o",
                            os.path.join(d, "t.o"), "-I", os.path.join(ROOT, "include"),
                            "-I", "/usr/local/cuda/include"], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_abi_version_and_status_strings():
    assert _abi.lib.ccc_conv1d_abi_version() == _abi.ABI_VERSION
    for code in range(10):
        assert _abi.status_string(code) != "unknown status"
    assert _abi.status_string(99) == "unknown status"


# ---- fake descriptors --------------------------------------------------------

_BASE = 0x7f0000000000


def T(addr_off, dtype, shape, stride=None):
    d = _abi.ccc_tensor()
    d.data = _BASE + addr_off
    d.dtype = dtype
    d.ndim = len(shape)
    if stride is None:  # contiguous
        stride, s = [], 1
        for n in reversed(shape):
            stride.insert(0, s)
            s *= n
    for i, (n, st) in enumerate(zip(shape, stride)):
        d.shape[i] = n
        d.stride[i] = st
    return d


def cl(off, B, D, Tn):
    """Channel-last [B, D, T] view of [B, T, D] storage."""
    return T(off, BF16, (B, D, Tn), (Tn * D, 1, D))


MB = 1 << 20


def fwd(x, w, b=None, cu=None, init=None, out=None, fin=None, act=1, ids=None):
    r = lambda d: None if d is None else ctypes.byref(d)
    return _abi.lib.ccc_conv1d_fwd(r(x), r(w), r(b), r(cu), r(ids), r(init), r(out), r(fin), act,
                                   None, None)


def bwd(x, w, b, cu, init, g, gf, dx, dw, db, dinit, det=0, act=1, ws=None, ws_bytes=0, ids=None):
    r = lambda d: None if d is None else ctypes.byref(d)
    return _abi.lib.ccc_conv1d_bwd(r(x), r(w), r(b), r(cu), r(ids), r(init), r(g), r(gf), r(dx),
                                   r(dw), r(db), r(dinit), act, det, ws, ws_bytes, None, None)


B_, D_, T_ = 2, 16, 32


def good():
    return dict(x=cl(0, B_, D_, T_), w=T(10 * MB, BF16, (D_, 4)), b=T(11 * MB, BF16, (D_,)),
                init=T(12 * MB, BF16, (B_, D_, 3)), out=cl(20 * MB, B_, D_, T_),
                fin=T(30 * MB, BF16, (B_, D_, 3)))


def test_fwd_rejects_bad_arguments_on_host():
    g = good()
    bad_x = cl(0, B_, D_, T_)
    bad_x.dtype = F32
    assert fwd(bad_x, g["w"], out=g["out"]) == _abi.CCC_ERR_INVALID_ARG
    # widths 2..4 are served; 1 and 5 decline
    assert fwd(g["x"], T(10 * MB, BF16, (D_, 5)), out=g["out"]) == _abi.CCC_ERR_UNSUPPORTED
    assert fwd(g["x"], T(10 * MB, BF16, (D_, 1)), out=g["out"]) == _abi.CCC_ERR_UNSUPPORTED
    # a width-3 weight takes [S, D, 2] states
    assert fwd(g["x"], T(10 * MB, BF16, (D_, 3)), init=g["init"], out=g["out"]) == _abi.CCC_ERR_INVALID_ARG
    assert fwd(g["x"], T(10 * MB, BF16, (D_ + 1, 4)), out=g["out"]) == _abi.CCC_ERR_INVALID_ARG
    # FP32 weight with bias declines (cuDNN page)
    assert fwd(g["x"], T(10 * MB, F32, (D_, 4)), g["b"], out=g["out"]) == _abi.CCC_ERR_UNSUPPORTED
    # unknown activation
    assert fwd(g["x"], g["w"], out=g["out"], act=7) == _abi.CCC_ERR_INVALID_ARG
    # neither channel-last nor time-contiguous
    odd = T(0, BF16, (B_, D_, T_), (D_ * T_ * 4, 2, 2 * D_))
    assert fwd(odd, g["w"], out=cl(20 * MB, B_, D_, T_)) == _abi.CCC_ERR_UNSUPPORTED
    # out with a different layout kind than x
    assert fwd(g["x"], g["w"], out=T(20 * MB, BF16, (B_, D_, T_))) == _abi.CCC_ERR_UNSUPPORTED
    # states: wrong shape, non-contiguous
    assert fwd(g["x"], g["w"], init=T(12 * MB, BF16, (B_, D_, 4)), out=g["out"]) == _abi.CCC_ERR_INVALID_ARG
    assert fwd(g["x"], g["w"], out=g["out"],
               fin=T(30 * MB, BF16, (B_, D_, 3), (D_ * 3, 1, D_))) == _abi.CCC_ERR_INVALID_ARG
    # packed with batch 2
    cu = T(40 * MB, I32, (3,))
    assert fwd(g["x"], g["w"], cu=cu, out=g["out"]) == _abi.CCC_ERR_UNSUPPORTED
    # NULL x
    assert fwd(None, g["w"], out=g["out"]) == _abi.CCC_ERR_INVALID_ARG


@pytest.mark.parametrize("victim", ["x", "w", "b", "init", "cu"])
def test_fwd_final_states_aliasing_is_rejected(victim):
    """cuDNN page: final_states_out must not share memory with x, weight, bias,
    cu_seqlens or initial_states."""
    g = good()
    x = cl(0, 1, D_, T_)
    cu = T(40 * MB, I32, (3,))
    init = T(12 * MB, BF16, (2, D_, 3))
    out = cl(20 * MB, 1, D_, T_)
    addr = {"x": 0, "w": 10 * MB, "b": 11 * MB, "init": 12 * MB, "cu": 40 * MB}[victim]
    fin = T(addr, BF16, (2, D_, 3))
    assert fwd(x, g["w"], g["b"], cu, init, out, fin) == _abi.CCC_ERR_ALIAS


def test_fwd_out_overlapping_input_is_rejected():
    g = good()
    assert fwd(g["x"], g["w"], g["b"], None, g["init"], cl(64, B_, D_, T_), g["fin"]) == _abi.CCC_ERR_ALIAS


def test_bwd_rejects_bad_arguments_on_host():
    g = good()
    dout = cl(50 * MB, B_, D_, T_)
    dx = cl(60 * MB, B_, D_, T_)
    dw = T(70 * MB, BF16, (D_, 4))
    db = T(71 * MB, BF16, (D_,))
    dinit = T(72 * MB, BF16, (B_, D_, 3))
    # deterministic with bias: no deterministic dbias route (cuDNN page)
    assert bwd(g["x"], g["w"], g["b"], None, g["init"], dout, None, dx, dw, db, dinit,
               det=1) == _abi.CCC_ERR_NONDETERMINISTIC
    # dbias required iff bias
    assert bwd(g["x"], g["w"], g["b"], None, g["init"], dout, None, dx, dw, None, dinit) == _abi.CCC_ERR_INVALID_ARG
    assert bwd(g["x"], g["w"], None, None, g["init"], dout, None, dx, dw, db, dinit) == _abi.CCC_ERR_INVALID_ARG
    # dweight dtype must follow weight
    assert bwd(g["x"], g["w"], g["b"], None, g["init"], dout, None, dx,
               T(70 * MB, F32, (D_, 4)), db, dinit) == _abi.CCC_ERR_INVALID_ARG
    # dinitial_states without initial_states
    assert bwd(g["x"], g["w"], g["b"], None, None, dout, None, dx, dw, db, dinit) == _abi.CCC_ERR_INVALID_ARG
    # dx overlapping dout
    assert bwd(g["x"], g["w"], g["b"], None, g["init"], dout, None, cl(50 * MB + 2, B_, D_, T_), dw,
               db, dinit) == _abi.CCC_ERR_ALIAS
    # dweight overlapping dbias
    assert bwd(g["x"], g["w"], g["b"], None, g["init"], dout, None, dx, dw,
               T(70 * MB + 8, BF16, (D_,)), dinit) == _abi.CCC_ERR_ALIAS
    assert bwd(g["x"], g["w"], g["b"], None, g["init"], dout, None, dx, dw, db, dinit,
               det=2) == _abi.CCC_ERR_INVALID_ARG


def test_seq_idx_host_checks():
    """seq_idx [B, T] int32: mutually exclusive with cu_seqlens (cuDNN page),
    no state with it, outputs may not overlap it."""
    g = good()
    ids = T(80 * MB, I32, (B_, T_))
    dout = cl(50 * MB, B_, D_, T_)
    dx = cl(60 * MB, B_, D_, T_)
    dw = T(70 * MB, BF16, (D_, 4))
    db = T(71 * MB, BF16, (D_,))
    # wrong shape or dtype
    assert fwd(g["x"], g["w"], g["b"], out=g["out"], ids=T(80 * MB, I32, (B_, T_ + 1))) == _abi.CCC_ERR_INVALID_ARG
    assert fwd(g["x"], g["w"], g["b"], out=g["out"], ids=T(80 * MB, BF16, (B_, T_))) == _abi.CCC_ERR_INVALID_ARG
    # with cu_seqlens
    x1, out1 = cl(0, 1, D_, T_), cl(20 * MB, 1, D_, T_)
    assert fwd(x1, g["w"], g["b"], cu=T(40 * MB, I32, (3,)), out=out1,
               ids=T(80 * MB, I32, (1, T_))) == _abi.CCC_ERR_INVALID_ARG
    # no state with seq_idx
    assert fwd(g["x"], g["w"], g["b"], init=g["init"], out=g["out"], ids=ids) == _abi.CCC_ERR_UNSUPPORTED
    assert fwd(g["x"], g["w"], g["b"], out=g["out"], fin=g["fin"], ids=ids) == _abi.CCC_ERR_UNSUPPORTED
    assert bwd(g["x"], g["w"], g["b"], None, None, dout, T(90 * MB, BF16, (B_, D_, 3)), dx, dw, db,
               None, ids=ids) == _abi.CCC_ERR_UNSUPPORTED
    # outputs overlapping the ids
    assert fwd(g["x"], g["w"], g["b"], out=cl(80 * MB, B_, D_, T_), ids=ids) == _abi.CCC_ERR_ALIAS
    assert bwd(g["x"], g["w"], g["b"], None, None, dout, None, cl(80 * MB, B_, D_, T_), dw, db,
               None, ids=ids) == _abi.CCC_ERR_ALIAS


def test_update_rejects_bad_arguments_on_host():
    r = lambda d: None if d is None else ctypes.byref(d)
    x = T(0, BF16, (4, D_))
    st = T(MB, BF16, (4, D_, 3))
    w = T(2 * MB, BF16, (D_, 4))
    b = T(3 * MB, BF16, (D_,))
    out = T(4 * MB, BF16, (4, D_))
    upd = lambda *a, act=1: _abi.lib.ccc_conv1d_update(*[r(d) for d in a], act, None)
    assert upd(x, T(MB, BF16, (4, D_, 4)), w, b, out) == _abi.CCC_ERR_INVALID_ARG
    assert upd(x, st, w, b, T(MB + 6, BF16, (4, D_))) == _abi.CCC_ERR_ALIAS  # out on the state
    assert upd(T(MB, BF16, (4, D_)), st, w, b, out) == _abi.CCC_ERR_ALIAS    # x on the state
    assert upd(x, st, T(2 * MB, F32, (D_, 4)), b, out) == _abi.CCC_ERR_UNSUPPORTED
    assert upd(T(0, BF16, (4, D_), (1, 4)), st, w, b, out) == _abi.CCC_ERR_UNSUPPORTED


def test_multi_token_update_host_checks():
    """x [B, D, L]: out must have x's rank and shape, channel stride 1, and may
    be x itself but not a shifted view of it; L == 0 is a no-op that touches
    no memory (the fake pointers here are never dereferenced)."""
    r = lambda d: None if d is None else ctypes.byref(d)
    upd = lambda *a, act=1: _abi.lib.ccc_conv1d_update(*[r(d) for d in a], act, None)
    L = 5
    cl3 = lambda off, Ln=L: T(off, BF16, (4, D_, Ln), (Ln * D_, 1, D_))  # [B, L, D] storage
    st = T(MB, BF16, (4, D_, 3))
    w = T(2 * MB, BF16, (D_, 4))
    b = T(3 * MB, BF16, (D_,))
    x = cl3(0)
    # rank or shape mismatch between x and out
    assert upd(x, st, w, b, T(4 * MB, BF16, (4, D_))) == _abi.CCC_ERR_INVALID_ARG
    assert upd(x, st, w, b, cl3(4 * MB, L + 1)) == _abi.CCC_ERR_INVALID_ARG
    # time-contiguous x or out (channel stride != 1) is declined: the wrapper restrides
    assert upd(T(0, BF16, (4, D_, L)), st, w, b, cl3(4 * MB)) == _abi.CCC_ERR_UNSUPPORTED
    assert upd(x, st, w, b, T(4 * MB, BF16, (4, D_, L))) == _abi.CCC_ERR_UNSUPPORTED
    # out a shifted view of x: another thread's tokens would be overwritten
    assert upd(x, st, w, b, cl3(2 * D_)) == _abi.CCC_ERR_ALIAS
    # out on the state
    assert upd(x, st, w, b, cl3(MB)) == _abi.CCC_ERR_ALIAS
    # no tokens: nothing to do, nothing touched
    assert upd(cl3(0, 0), st, w, b, cl3(4 * MB, 0)) == _abi.CCC_OK


def test_python_api_seq_idx_rules_and_bad_activation():
    import torch

    x = torch.zeros(1, 8, 4, dtype=torch.bfloat16)
    w = torch.zeros(8, 4, dtype=torch.bfloat16)
    ids = torch.zeros(1, 4, dtype=torch.int32)
    with pytest.raises(ValueError):       # int32 only
        ccc.causal_conv1d(x, w, seq_idx=ids.long())
    with pytest.raises(ValueError):       # mutually exclusive with cu_seqlens
        ccc.causal_conv1d(x, w, seq_idx=ids, cu_seqlens=torch.tensor([0, 4], dtype=torch.int32))
    with pytest.raises(NotImplementedError):  # no state with seq_idx
        ccc.causal_conv1d(x, w, seq_idx=ids, initial_states=torch.zeros(1, 8, 3, dtype=torch.bfloat16))
    with pytest.raises(NotImplementedError):
        ccc.causal_conv1d(x, w, seq_idx=ids, return_final_states=True)
    with pytest.raises(ValueError):
        ccc.causal_conv1d(x, w, activation="gelu")


def fc(x, pw, b, dil, out):
    r = lambda d: None if d is None else ctypes.byref(d)
    return _abi.lib.ccc_fullconv1d_fwd(r(x), r(pw), r(b), int(dil), r(out), None, None)


def test_fullconv_rejects_bad_arguments_on_host():
    """ccc_fullconv1d_fwd and ccc_fullconv1d_pack_weight: every call below
    fails a host-side check before the first CUDA call."""
    B, Cin, Cout, Tn, K = 2, 64, 96, 40, 3
    x = cl(0, B, Cin, Tn)
    pw = T(10 * MB, BF16, (K, Cout, Cin))
    b = T(11 * MB, BF16, (Cout,))
    out = cl(20 * MB, B, Cout, Tn)
    inv, uns, ali = _abi.CCC_ERR_INVALID_ARG, _abi.CCC_ERR_UNSUPPORTED, _abi.CCC_ERR_ALIAS
    assert fc(x, pw, b, 0, out) == inv                                   # dilation >= 1
    assert fc(x, T(10 * MB, BF16, (K, Cout, Cin + 8)), b, 1, out) == inv  # Cin of x and weight differ
    assert fc(x, pw, T(11 * MB, BF16, (Cout + 8,)), 1, out) == inv       # bias shape
    assert fc(x, pw, b, 1, cl(20 * MB, B, Cout, Tn + 1)) == inv          # out shape
    assert fc(x, pw, b, 1, T(20 * MB, F32, (B, Cout, Tn), (Tn * Cout, 1, Cout))) == inv  # out dtype
    xt = T(0, BF16, (B, Cin, Tn))                                        # time-contiguous x
    assert fc(xt, pw, b, 1, out) == uns
    x60 = cl(0, B, 60, Tn)                                               # Cin not a multiple of 8
    assert fc(x60, T(10 * MB, BF16, (K, Cout, 60)), b, 1, out) == uns
    assert fc(x, T(10 * MB, BF16, (1025, Cout, Cin)), b, 1, out) == uns  # K above 1024
    assert fc(x, pw, b, 1, cl(0, B, Cout, Tn)) == ali                    # out on top of x
    assert fc(x, pw, b, 1, cl(10 * MB, B, Cout, Tn)) == ali              # out on top of the weight
    # more 256 x 256 tiles than the persistent kernel numbers (2^31 here)
    Bb, Tb, Cb = 4096, 1 << 24, 2048
    xb = cl(0, Bb, Cin, Tb)
    ob = T(1 << 50, BF16, (Bb, Cb, Tb), (Tb * Cb, 1, Cb))
    assert fc(xb, T(1 << 49, BF16, (K, Cb, Cin)), None, 1, ob) == uns
    # the pack: contiguous packed output, no overlap with the weight
    w = T(40 * MB, BF16, (Cout, Cin, K))
    r = lambda d: ctypes.byref(d)
    assert _abi.lib.ccc_fullconv1d_pack_weight(r(w), r(T(50 * MB, BF16, (K, Cout, Cin + 8))), None) == inv
    assert _abi.lib.ccc_fullconv1d_pack_weight(
        r(w), r(T(50 * MB, BF16, (K, Cout, Cin), (Cout * Cin * 2, Cin, 1))), None) == uns
    assert _abi.lib.ccc_fullconv1d_pack_weight(r(w), r(T(40 * MB, BF16, (K, Cout, Cin))), None) == ali
