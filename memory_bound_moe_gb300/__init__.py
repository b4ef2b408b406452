"""GB300 (sm_103a) memory-bound MoE glue path: route, expand, SwiGLU, combine.

Thin Python binding over the C ABI in ``include/moe_glue.h`` (library
``lib/libmoeglue.so``). The functions here only marshal arguments: they check
tensor dtypes, shapes and devices, allocate outputs with PyTorch when none are
given, and call the C entry point of the same name on the current CUDA
stream. Every step of the path runs in the library's kernels; there is no
Python or CPU fallback, and a missing library is an error.
"""
from __future__ import annotations

from .binding import (MoeError, RouteResult, STATUS, library_path, load_library, moe_combine,
                      moe_combine_rows, moe_expand, moe_expand_rows, moe_route, moe_route_expand,
                      moe_route_local, moe_route_local_rows, moe_route_local_workspace_size,
                      moe_route_workspace_size, moe_status_string, moe_swiglu,
                      moe_swiglu_mxfp8, moe_expand_mxfp8, moe_swiglu_fp4, moe_expand_fp4,
                      moe_qk_rmsnorm)

__all__ = ["MoeError", "RouteResult", "STATUS", "library_path", "load_library", "moe_combine",
           "moe_combine_rows", "moe_expand", "moe_expand_rows", "moe_route", "moe_route_expand",
           "moe_route_local", "moe_route_local_rows", "moe_route_local_workspace_size",
           "moe_route_workspace_size", "moe_status_string", "moe_swiglu",
           "moe_swiglu_mxfp8", "moe_expand_mxfp8", "moe_swiglu_fp4", "moe_expand_fp4", "moe_qk_rmsnorm"]
