"""Depthwise causal conv1d for GB300 (sm_103a): BF16 activations, filter
widths 2..4, SiLU, W-1 initial/final state, cu_seqlens packing, per-token
sequence ids (seq_idx), backward, and the in-place decode update of one or
several tokens -- as hand-written CUDA kernels behind a C ABI
(include/ccc_conv1d.h, libccc_conv1d.so).  Also the full-channel dilated
causal conv1d (forward) on the tensor cores.

``causal_conv1d``, ``causal_conv1d_update`` and ``full_causal_conv1d`` are the
model-facing calls; ``_abi`` holds the ctypes binding with the C function
names.  Importing this package loads the CUDA library and raises ImportError
when it has not been built: there is no fallback path.
"""

from . import _abi
from ._abi import Conv1dError
from .functional import (causal_conv1d, causal_conv1d_update, check_status, full_causal_conv1d,
                         pack_full_conv_weight, status_word)

__all__ = ["causal_conv1d", "causal_conv1d_update", "full_causal_conv1d", "pack_full_conv_weight",
           "check_status", "status_word", "Conv1dError", "_abi"]
