"""ctypes binding of the C ABI in include/ccc_conv1d.h (libccc_conv1d.so).

Argument marshalling only: each function takes torch tensors (or None), builds
the ccc_tensor descriptors (data pointer, dtype, shape, strides in elements)
and calls the library function of the same name on the given CUDA stream.  All
computation happens in the library's kernels.  The library must be built
(``build.build()``); importing this module on a machine without it raises.
"""

from __future__ import annotations

import ctypes
import os
import struct

import torch

from . import build as _build

CCC_OK = 0
CCC_ERR_INVALID_ARG = 1
CCC_ERR_UNSUPPORTED = 2
CCC_ERR_ALIAS = 3
CCC_ERR_NONDETERMINISTIC = 4
CCC_ERR_WORKSPACE = 5
CCC_ERR_CUDA = 6
CCC_ERR_BAD_CU_SEQLENS = 7
CCC_ERR_SCRATCH_LIMIT = 8
CCC_ERR_DEVICE_TIMEOUT = 9

CCC_BF16, CCC_F32, CCC_I32 = 0, 1, 2
CCC_ACT_NONE, CCC_ACT_SILU = 0, 1

ABI_VERSION = 2

EXPORTED = (
    "ccc_conv1d_fwd",
    "ccc_conv1d_bwd_workspace_size",
    "ccc_conv1d_bwd",
    "ccc_conv1d_bwd_noalloc",
    "ccc_conv1d_update",
    "ccc_fullconv1d_pack_weight",
    "ccc_fullconv1d_fwd",
    "ccc_read_status",
    "ccc_status_string",
    "ccc_conv1d_abi_version",
)

_DTYPES = {torch.bfloat16: CCC_BF16, torch.float32: CCC_F32, torch.int32: CCC_I32}


class ccc_tensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 3),
        ("stride", ctypes.c_int64 * 3),
    ]


class Conv1dError(RuntimeError):
    """A non-OK ccc_status from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(ccc_tensor)
    V = ctypes.c_void_p
    I = ctypes.c_int
    lib.ccc_conv1d_fwd.argtypes = [P, P, P, P, P, P, P, P, I, V, V]
    lib.ccc_conv1d_fwd.restype = I
    lib.ccc_conv1d_bwd_workspace_size.argtypes = [P, I]
    lib.ccc_conv1d_bwd_workspace_size.restype = ctypes.c_size_t
    lib.ccc_conv1d_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, V, ctypes.c_size_t, V, V]
    lib.ccc_conv1d_bwd.restype = I
    lib.ccc_conv1d_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, V, V]
    lib.ccc_conv1d_bwd_noalloc.restype = I
    lib.ccc_conv1d_update.argtypes = [P, P, P, P, P, I, V]
    lib.ccc_conv1d_update.restype = I
    lib.ccc_fullconv1d_pack_weight.argtypes = [P, P, V]
    lib.ccc_fullconv1d_pack_weight.restype = I
    lib.ccc_fullconv1d_fwd.argtypes = [P, P, P, I, P, V, V]
    lib.ccc_fullconv1d_fwd.restype = I
    lib.ccc_read_status.argtypes = [V, V]
    lib.ccc_read_status.restype = I
    lib.ccc_status_string.argtypes = [I]
    lib.ccc_status_string.restype = ctypes.c_char_p
    lib.ccc_conv1d_abi_version.argtypes = []
    lib.ccc_conv1d_abi_version.restype = I
    if lib.ccc_conv1d_abi_version() != ABI_VERSION:
        raise ImportError(f"{path}: ABI version {lib.ccc_conv1d_abi_version()} != {ABI_VERSION}")
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.ccc_status_string(int(status)).decode()


_PACK = struct.Struct("<Qii3q3q")  # the ccc_tensor layout: 64 bytes
_desc_memo = {}


def desc(t):
    """ccc_tensor descriptor of a torch tensor, or None.  Descriptors are a pure
    function of (address, dtype, shape, strides) and are memoised on that key."""
    if t is None:
        return None
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    d = _desc_memo.get(key)
    if d is not None:
        return d
    code = _DTYPES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    n = t.dim()
    if n > 3:
        raise ValueError("tensors have at most 3 dimensions")
    pad = (0,) * (3 - n)
    d = ccc_tensor.from_buffer_copy(_PACK.pack(t.data_ptr() if t.numel() > 0 else 0, code, n,
                                               *tuple(t.shape), *pad, *t.stride(), *pad))
    if len(_desc_memo) > 4096:
        _desc_memo.clear()
    _desc_memo[key] = d
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _status_ptr(status):
    return None if status is None else status.data_ptr()


def ccc_conv1d_fwd(x, weight, bias, cu_seqlens, initial_states, out, final_states,
                   activation: int, status=None, stream=None, seq_idx=None) -> int:
    ds = [desc(t) for t in (x, weight, bias, cu_seqlens, seq_idx, initial_states, out,
                            final_states)]
    return lib.ccc_conv1d_fwd(*[_ref(d) for d in ds], int(activation), _status_ptr(status),
                              _stream(stream))


def ccc_conv1d_bwd_workspace_size(x, deterministic: bool) -> int:
    return int(lib.ccc_conv1d_bwd_workspace_size(_ref(desc(x)), int(bool(deterministic))))


def ccc_conv1d_bwd(x, weight, bias, cu_seqlens, initial_states, dout, dfinal_states, dx,
                   dweight, dbias, dinitial_states, activation: int, deterministic: bool,
                   workspace, status=None, stream=None, seq_idx=None) -> int:
    ds = [desc(t) for t in (x, weight, bias, cu_seqlens, seq_idx, initial_states, dout,
                            dfinal_states, dx, dweight, dbias, dinitial_states)]
    ws_ptr = workspace.data_ptr() if workspace is not None and workspace.numel() > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return lib.ccc_conv1d_bwd(*[_ref(d) for d in ds], int(activation), int(bool(deterministic)),
                              ws_ptr, ws_bytes, _status_ptr(status), _stream(stream))


def ccc_conv1d_bwd_noalloc(x, weight, bias, cu_seqlens, initial_states, dout, dfinal_states,
                           dx, dweight, dbias, dinitial_states, activation: int,
                           deterministic: bool, status=None, stream=None) -> int:
    """ccc_conv1d_bwd with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    ds = [desc(t) for t in (x, weight, bias, cu_seqlens, initial_states, dout, dfinal_states,
                            dx, dweight, dbias, dinitial_states)]
    return lib.ccc_conv1d_bwd_noalloc(*[_ref(d) for d in ds], int(activation),
                                      int(bool(deterministic)), _status_ptr(status),
                                      _stream(stream))


def ccc_conv1d_update(x, conv_state, weight, bias, out, activation: int, stream=None) -> int:
    ds = [desc(t) for t in (x, conv_state, weight, bias, out)]
    return lib.ccc_conv1d_update(*[_ref(d) for d in ds], int(activation), _stream(stream))


def ccc_fullconv1d_pack_weight(weight, packed, stream=None) -> int:
    return lib.ccc_fullconv1d_pack_weight(_ref(desc(weight)), _ref(desc(packed)), _stream(stream))


def ccc_fullconv1d_fwd(x, packed_weight, bias, dilation: int, out, status=None, stream=None) -> int:
    ds = [desc(t) for t in (x, packed_weight, bias)]
    return lib.ccc_fullconv1d_fwd(*[_ref(d) for d in ds], int(dilation), _ref(desc(out)),
                                  _status_ptr(status), _stream(stream))


def ccc_read_status(status, stream=None) -> int:
    return lib.ccc_read_status(_status_ptr(status), _stream(stream))
