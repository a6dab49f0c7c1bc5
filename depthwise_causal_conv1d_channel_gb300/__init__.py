"""Depthwise causal conv1d for GB300 (sm_103a): BF16 activations, filter
widths 2..4, SiLU, W-1 initial/final state, cu_seqlens packing, backward, and
the in-place decode update of one or several tokens -- as hand-written CUDA
kernels behind a C ABI (include/ccc_conv1d.h, libccc_conv1d.so).

``causal_conv1d`` and ``causal_conv1d_update`` are the model-facing calls;
``_abi`` holds the ctypes binding with the C function names.  Importing this
package loads the CUDA library and raises ImportError when it has not been
built: there is no fallback path.
"""

from . import _abi
from ._abi import Conv1dError
from .functional import causal_conv1d, causal_conv1d_update, check_status, status_word

__all__ = ["causal_conv1d", "causal_conv1d_update", "check_status", "status_word", "Conv1dError",
           "_abi"]
