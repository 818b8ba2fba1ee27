"""quantized_q4_q8_gb300 -- GB300-native Q4_K x Q8_1 single-token decode.

The compute lives in librz (CUDA for sm_103a, C ABI in include/rz.h).  This
package is its Python binding: torch supplies device memory and streams, every
step runs in librz's kernels.  Functions named rz_* take raw device pointers and
sizes exactly like the C entry points; the lower-case helpers take torch CUDA
tensors, allocate the outputs with torch and call the same entry points.
"""
from __future__ import annotations

from . import _lib
from ._lib import RzError, call, load  # noqa: F401
from .ops import *  # noqa: F401,F403
from .ops import __all__ as _ops_all

__all__ = ["RzError", "load", "build"] + list(_ops_all)


def build(force: bool = False, verbose: bool = False) -> str:
    from .build import build as _build
    return _build(force=force, verbose=verbose)
