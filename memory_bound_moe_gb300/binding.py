"""ctypes binding of ``libmoeglue.so`` (see ``include/moe_glue.h``).

Argument marshalling only: tensors are checked, outputs allocated on the
tensors' device when not supplied, and the raw device pointers plus the
current CUDA stream are passed to the C entry point. The library is loaded
lazily on first use; if it has not been built the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libmoeglue.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_MISALIGNED",
          3: "MOE_ERR_UNSUPPORTED", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA"}

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


class MoeError(RuntimeError):
    """A non-OK status from the C library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``libmoeglue.so`` (once). Raises if it is missing: build it with
    ``memory_bound_moe_gb300.build.build()``."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_LIB_PATH} is missing "
                               "(run memory_bound_moe_gb300.build.build())")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.moe_status_string.argtypes = [_int]
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_route_workspace_size.argtypes = [_i64, _int, _int, ctypes.POINTER(ctypes.c_size_t)]
        lib.moe_route_workspace_size.restype = _int
        lib.moe_route.argtypes = [_vp, _i64, _int, _int, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, ctypes.c_size_t, _vp]
        lib.moe_route.restype = _int
        lib.moe_route_expand.argtypes = [_vp, _i64, _int, _int, _int, _vp, _int, _vp, _vp, _vp,
                                         _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.moe_route_expand.restype = _int
        lib.moe_route_local_rows.argtypes = [_i64, _int, _int, _int, _int, ctypes.POINTER(_i64)]
        lib.moe_route_local_rows.restype = _int
        lib.moe_route_local_workspace_size.argtypes = [_i64, _int, _int, _int, _int,
                                                       ctypes.POINTER(ctypes.c_size_t)]
        lib.moe_route_local_workspace_size.restype = _int
        lib.moe_route_local.argtypes = [_vp, _i64, _int, _int, _int, _int, _int, _int, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.moe_route_local.restype = _int
        lib.moe_expand_rows.argtypes = [_vp, _i64, _int, _int, _vp, _i64, _vp, _vp]
        lib.moe_expand_rows.restype = _int
        lib.moe_combine_rows.argtypes = [_vp, _i64, _i64, _int, _int, _vp, _vp, _vp, _vp]
        lib.moe_combine_rows.restype = _int
        lib.moe_swiglu_mxfp8.argtypes = [_vp, _i64, _int, _vp, _vp, _vp]
        lib.moe_swiglu_mxfp8.restype = _int
        lib.moe_expand_mxfp8.argtypes = [_vp, _i64, _int, _int, _vp, _i64, _vp, _vp, _vp]
        lib.moe_expand_mxfp8.restype = _int
        lib.moe_swiglu_fp4.argtypes = [_vp, _i64, _int, _int, ctypes.c_float, _vp, _vp, _vp]
        lib.moe_swiglu_fp4.restype = _int
        lib.moe_expand_fp4.argtypes = [_vp, _i64, _int, _int, _vp, _i64, _int, ctypes.c_float, _vp, _vp, _vp]
        lib.moe_expand_fp4.restype = _int
        lib.moe_qk_rmsnorm.argtypes = [_vp, _vp, _i64, _int, _int, _int, _vp, _vp, ctypes.c_float,
                                       ctypes.c_float, _vp]
        lib.moe_qk_rmsnorm.restype = _int
        lib.moe_expand.argtypes = [_vp, _i64, _int, _int, _vp, _vp, _vp]
        lib.moe_expand.restype = _int
        lib.moe_swiglu.argtypes = [_vp, _i64, _int, _vp, _vp]
        lib.moe_swiglu.restype = _int
        lib.moe_combine.argtypes = [_vp, _i64, _int, _int, _vp, _vp, _vp, _vp]
        lib.moe_combine.restype = _int
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != 0:
        raise MoeError(fn, status)


def _stream_ptr(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None or t.numel() == 0 else t.data_ptr()


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def moe_route_workspace_size(T: int, E: int, k: int) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_route_workspace_size",
           load_library().moe_route_workspace_size(int(T), int(E), int(k), ctypes.byref(out)))
    return out.value


class RouteResult(NamedTuple):
    topk_ids: torch.Tensor        # [T, k] int32
    topk_weights: torch.Tensor    # [T, k] float32
    expert_counts: torch.Tensor   # [E] int32
    expert_offsets: torch.Tensor  # [E + 1] int32
    perm: torch.Tensor            # [T*k] int32, sorted row -> flat slot
    inv_perm: torch.Tensor        # [T*k] int32, flat slot -> sorted row


def moe_route(logits: torch.Tensor, k: int, renorm: bool, *, out: Optional[RouteResult] = None,
              workspace: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None) -> RouteResult:
    """Top-k routing and the expert-sorted permutation of ``logits [T, E]``
    (float32). ``workspace`` is a uint8 CUDA tensor of at least
    ``moe_route_workspace_size(T, E, k)`` bytes (allocated when omitted)."""
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    _need(logits, "logits", torch.float32, (T, E))
    dev = logits.device
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = RouteResult(torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev),
                          torch.empty((E,), **i32), torch.empty((E + 1,), **i32),
                          torch.empty((T * k,), **i32), torch.empty((T * k,), **i32))
    _need(out.topk_ids, "topk_ids", torch.int32, (T, k))
    _need(out.topk_weights, "topk_weights", torch.float32, (T, k))
    _need(out.expert_counts, "expert_counts", torch.int32, (E,))
    _need(out.expert_offsets, "expert_offsets", torch.int32, (E + 1,))
    _need(out.perm, "perm", torch.int32, (T * k,))
    _need(out.inv_perm, "inv_perm", torch.int32, (T * k,))
    ws_bytes = moe_route_workspace_size(T, E, k)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    if workspace is not None:
        if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 CUDA tensor")
    ws_len = 0 if workspace is None else workspace.numel()
    st = load_library().moe_route(_ptr(logits), T, E, int(k), int(bool(renorm)),
                                  _ptr(out.topk_ids), _ptr(out.topk_weights),
                                  _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                  _ptr(out.perm), _ptr(out.inv_perm), _ptr(workspace), ws_len,
                                  _stream_ptr(stream, dev))
    _check("moe_route", st)
    return out


def _route_outputs(T: int, E: int, k: int, dev) -> RouteResult:
    i32 = dict(dtype=torch.int32, device=dev)
    return RouteResult(torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev),
                       torch.empty((E,), **i32), torch.empty((E + 1,), **i32),
                       torch.empty((T * k,), **i32), torch.empty((T * k,), **i32))


def moe_route_expand(logits: torch.Tensor, x: torch.Tensor, k: int, renorm: bool, *,
                     out: Optional[RouteResult] = None, expanded: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None):
    """Routing of ``logits [T, E]`` and expansion of ``x [T, H]`` in one call
    (one kernel launch for decode-sized T). Returns ``(RouteResult,
    expanded_x)``, identical to ``moe_route`` followed by ``moe_expand``."""
    if logits.dim() != 2 or x.dim() != 2:
        raise ValueError("logits must be [T, E] and x [T, H]")
    T, E = logits.shape
    H = x.shape[1]
    _need(logits, "logits", torch.float32, (T, E))
    _need(x, "x", torch.bfloat16, (T, H))
    dev = logits.device
    if out is None:
        out = _route_outputs(T, E, k, dev)
    if expanded is None:
        expanded = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    _need(expanded, "expanded_x", torch.bfloat16, (T * k, H))
    for name, t, dt, shape in (("topk_ids", out.topk_ids, torch.int32, (T, k)),
                               ("topk_weights", out.topk_weights, torch.float32, (T, k)),
                               ("expert_counts", out.expert_counts, torch.int32, (E,)),
                               ("expert_offsets", out.expert_offsets, torch.int32, (E + 1,)),
                               ("perm", out.perm, torch.int32, (T * k,)),
                               ("inv_perm", out.inv_perm, torch.int32, (T * k,))):
        _need(t, name, dt, shape)
    ws_bytes = moe_route_workspace_size(T, E, k)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    ws_len = 0 if workspace is None else workspace.numel()
    st = load_library().moe_route_expand(_ptr(logits), T, E, int(k), int(bool(renorm)), _ptr(x), H,
                                         _ptr(out.topk_ids), _ptr(out.topk_weights),
                                         _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                         _ptr(out.perm), _ptr(out.inv_perm), _ptr(expanded),
                                         _ptr(workspace), ws_len, _stream_ptr(stream, dev))
    _check("moe_route_expand", st)
    return out, expanded


def moe_expand(x: torch.Tensor, inv_perm: torch.Tensor, k: int, *,
               out: Optional[torch.Tensor] = None,
               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """``out[inv_perm[t*k + j]] = x[t]``: expert-sorted copy of ``x [T, H]``
    (bfloat16) into ``[T*k, H]``."""
    if x.dim() != 2:
        raise ValueError("x must be [T, H]")
    T, H = x.shape
    _need(x, "x", torch.bfloat16, (T, H))
    _need(inv_perm, "inv_perm", torch.int32, (T * k,))
    if out is None:
        out = torch.empty((T * k, H), dtype=torch.bfloat16, device=x.device)
    _need(out, "expanded_x", torch.bfloat16, (T * k, H))
    _check("moe_expand", load_library().moe_expand(_ptr(x), T, H, int(k), _ptr(inv_perm),
                                                   _ptr(out), _stream_ptr(stream, x.device)))
    return out


def moe_swiglu(gate_up: torch.Tensor, *, out: Optional[torch.Tensor] = None,
               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """``act = silu(gate) * up`` over ``gate_up [rows, 2I]`` (bfloat16; gate
    is the first half of each row)."""
    if gate_up.dim() != 2 or gate_up.shape[1] % 2:
        raise ValueError("gate_up must be [rows, 2I]")
    rows, two_i = gate_up.shape
    I = two_i // 2
    _need(gate_up, "gate_up", torch.bfloat16, (rows, two_i))
    if out is None:
        out = torch.empty((rows, I), dtype=torch.bfloat16, device=gate_up.device)
    _need(out, "act", torch.bfloat16, (rows, I))
    _check("moe_swiglu", load_library().moe_swiglu(_ptr(gate_up), rows, I, _ptr(out),
                                                   _stream_ptr(stream, gate_up.device)))
    return out


def moe_combine(expert_out: torch.Tensor, topk_weights: torch.Tensor, inv_perm: torch.Tensor, *,
                out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """``out[t] = sum_j w[t, j] * expert_out[inv_perm[t*k + j]]`` for
    ``expert_out [T*k, H]`` (bfloat16) and ``topk_weights [T, k]`` (float32)."""
    if topk_weights.dim() != 2 or expert_out.dim() != 2:
        raise ValueError("expert_out must be [T*k, H] and topk_weights [T, k]")
    T, k = topk_weights.shape
    H = expert_out.shape[1]
    _need(expert_out, "expert_out", torch.bfloat16, (T * k, H))
    _need(topk_weights, "topk_weights", torch.float32, (T, k))
    _need(inv_perm, "inv_perm", torch.int32, (T * k,))
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=expert_out.device)
    _need(out, "out", torch.bfloat16, (T, H))
    _check("moe_combine", load_library().moe_combine(_ptr(expert_out), T, H, int(k),
                                                     _ptr(topk_weights), _ptr(inv_perm), _ptr(out),
                                                     _stream_ptr(stream, expert_out.device)))
    return out


# ---------------------------------------------------------------------------
# local (one tensor-parallel rank's) routing with padded expert segments
# ---------------------------------------------------------------------------

def moe_route_local_rows(T: int, k: int, e0: int, e1: int, pad: int) -> int:
    """Rows of a padded local buffer (perm, expanded_x, expert_out)."""
    out = _i64(0)
    _check("moe_route_local_rows",
           load_library().moe_route_local_rows(int(T), int(k), int(e0), int(e1), int(pad),
                                               ctypes.byref(out)))
    return out.value


def moe_route_local_workspace_size(T: int, E: int, k: int, e0: int, e1: int) -> int:
    out = ctypes.c_size_t(0)
    _check("moe_route_local_workspace_size",
           load_library().moe_route_local_workspace_size(int(T), int(E), int(k), int(e0), int(e1),
                                                         ctypes.byref(out)))
    return out.value


def moe_route_local(logits: torch.Tensor, k: int, renorm: bool, e0: int, e1: int, pad: int = 1, *,
                    out: Optional[RouteResult] = None, workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> RouteResult:
    """Routing of ``logits [T, E]`` for the experts [e0, e1) of one rank,
    expert segments padded to a multiple of ``pad``. expert_counts has e1-e0
    entries, expert_offsets e1-e0+1, perm ``moe_route_local_rows(...)`` (-1 on
    padding rows), inv_perm T*k (-1 for slots of other ranks' experts)."""
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    _need(logits, "logits", torch.float32, (T, E))
    dev = logits.device
    n = e1 - e0
    rows = moe_route_local_rows(T, k, e0, e1, pad)
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = RouteResult(torch.empty((T, k), **i32), torch.empty((T, k), dtype=torch.float32, device=dev),
                          torch.empty((n,), **i32), torch.empty((n + 1,), **i32),
                          torch.empty((rows,), **i32), torch.empty((T * k,), **i32))
    for name, t, dt, shape in (("topk_ids", out.topk_ids, torch.int32, (T, k)),
                               ("topk_weights", out.topk_weights, torch.float32, (T, k)),
                               ("expert_counts", out.expert_counts, torch.int32, (n,)),
                               ("expert_offsets", out.expert_offsets, torch.int32, (n + 1,)),
                               ("perm", out.perm, torch.int32, (rows,)),
                               ("inv_perm", out.inv_perm, torch.int32, (T * k,))):
        _need(t, name, dt, shape)
    ws_bytes = moe_route_local_workspace_size(T, E, k, e0, e1)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=dev)
    ws_len = 0 if workspace is None else workspace.numel()
    st = load_library().moe_route_local(_ptr(logits), T, E, int(k), int(bool(renorm)), int(e0), int(e1),
                                        int(pad), _ptr(out.topk_ids), _ptr(out.topk_weights),
                                        _ptr(out.expert_counts), _ptr(out.expert_offsets),
                                        _ptr(out.perm), _ptr(out.inv_perm), _ptr(workspace), ws_len,
                                        _stream_ptr(stream, dev))
    _check("moe_route_local", st)
    return out


def moe_expand_rows(x: torch.Tensor, inv_perm: torch.Tensor, k: int, rows: int, *,
                    out: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """moe_expand into ``rows`` rows; inv_perm entries outside [0, rows) are
    skipped and rows nothing maps to are left as they are."""
    T, H = x.shape
    _need(x, "x", torch.bfloat16, (T, H))
    _need(inv_perm, "inv_perm", torch.int32, (T * k,))
    if out is None:
        out = torch.empty((rows, H), dtype=torch.bfloat16, device=x.device)
    _need(out, "expanded_x", torch.bfloat16, (rows, H))
    _check("moe_expand_rows", load_library().moe_expand_rows(_ptr(x), T, H, int(k), _ptr(inv_perm), rows,
                                                             _ptr(out), _stream_ptr(stream, x.device)))
    return out


def moe_combine_rows(expert_out: torch.Tensor, topk_weights: torch.Tensor, inv_perm: torch.Tensor, *,
                     out: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """moe_combine over an expert_out of any number of rows; inv_perm entries
    outside [0, rows) contribute nothing (a rank's partial sum)."""
    T, k = topk_weights.shape
    rows, H = expert_out.shape
    _need(expert_out, "expert_out", torch.bfloat16, (rows, H))
    _need(topk_weights, "topk_weights", torch.float32, (T, k))
    _need(inv_perm, "inv_perm", torch.int32, (T * k,))
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=expert_out.device)
    _need(out, "out", torch.bfloat16, (T, H))
    _check("moe_combine_rows", load_library().moe_combine_rows(_ptr(expert_out), rows, T, H, int(k),
                                                               _ptr(topk_weights), _ptr(inv_perm), _ptr(out),
                                                               _stream_ptr(stream, expert_out.device)))
    return out


# ---------------------------------------------------------------------------
# MXFP8 outputs (E4M3 codes, E8M0 scale per 32 values)
# ---------------------------------------------------------------------------

def moe_swiglu_mxfp8(gate_up: torch.Tensor, *, codes: Optional[torch.Tensor] = None,
                     scales: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None):
    """SwiGLU of ``gate_up [rows, 2I]`` quantized to MXFP8: returns
    ``(codes uint8 [rows, I], scales uint8 [rows, I/32])``."""
    rows, two_i = gate_up.shape
    I = two_i // 2
    _need(gate_up, "gate_up", torch.bfloat16, (rows, two_i))
    dev = gate_up.device
    if codes is None:
        codes = torch.empty((rows, I), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((rows, I // 32), dtype=torch.uint8, device=dev)
    _need(codes, "act_codes", torch.uint8, (rows, I))
    _need(scales, "act_scales", torch.uint8, (rows, I // 32))
    _check("moe_swiglu_mxfp8", load_library().moe_swiglu_mxfp8(_ptr(gate_up), rows, I, _ptr(codes),
                                                               _ptr(scales), _stream_ptr(stream, dev)))
    return codes, scales


def moe_expand_mxfp8(x: torch.Tensor, inv_perm: torch.Tensor, k: int, rows: Optional[int] = None, *,
                     codes: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None):
    """Expansion of ``x [T, H]`` quantized to MXFP8 into ``rows`` rows
    (default T*k): returns ``(codes uint8 [rows, H], scales uint8 [rows, H/32])``."""
    T, H = x.shape
    _need(x, "x", torch.bfloat16, (T, H))
    _need(inv_perm, "inv_perm", torch.int32, (T * k,))
    rows = T * k if rows is None else rows
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, H), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((rows, H // 32), dtype=torch.uint8, device=dev)
    _need(codes, "codes", torch.uint8, (rows, H))
    _need(scales, "scales", torch.uint8, (rows, H // 32))
    _check("moe_expand_mxfp8", load_library().moe_expand_mxfp8(_ptr(x), T, H, int(k), _ptr(inv_perm), rows,
                                                               _ptr(codes), _ptr(scales),
                                                               _stream_ptr(stream, dev)))
    return codes, scales


FP4_FORMATS = {"nvfp4": (0, 16), "mxfp4": (1, 32)}   # C-ABI format code, values per scale


def _fp4(fmt: str):
    if fmt not in FP4_FORMATS:
        raise ValueError(f"unknown FP4 format {fmt!r}: expected one of {sorted(FP4_FORMATS)}")
    return FP4_FORMATS[fmt]


def moe_swiglu_fp4(gate_up: torch.Tensor, fmt: str = "nvfp4", global_scale: float = 1.0, *,
                   codes: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """SwiGLU of ``gate_up [rows, 2I]`` quantized to NVFP4 (tensor scale
    ``global_scale``) or MXFP4: returns ``(codes uint8 [rows, I/2], two per
    byte, scales uint8 [rows, I/16] E4M3 or [rows, I/32] E8M0)``."""
    code, block = _fp4(fmt)
    rows, two_i = gate_up.shape
    I = two_i // 2
    _need(gate_up, "gate_up", torch.bfloat16, (rows, two_i))
    dev = gate_up.device
    if codes is None:
        codes = torch.empty((rows, I // 2), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((rows, I // block), dtype=torch.uint8, device=dev)
    _need(codes, "act_codes", torch.uint8, (rows, I // 2))
    _need(scales, "act_scales", torch.uint8, (rows, I // block))
    _check("moe_swiglu_fp4", load_library().moe_swiglu_fp4(_ptr(gate_up), rows, I, code, float(global_scale),
                                                           _ptr(codes), _ptr(scales), _stream_ptr(stream, dev)))
    return codes, scales


def moe_expand_fp4(x: torch.Tensor, inv_perm: torch.Tensor, k: int, fmt: str = "nvfp4",
                   global_scale: float = 1.0, rows: Optional[int] = None, *,
                   codes: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """Expansion of ``x [T, H]`` quantized to NVFP4 or MXFP4 into ``rows``
    rows (default T*k): returns ``(codes uint8 [rows, H/2], scales uint8
    [rows, H/16] or [rows, H/32])``."""
    code, block = _fp4(fmt)
    T, H = x.shape
    _need(x, "x", torch.bfloat16, (T, H))
    _need(inv_perm, "inv_perm", torch.int32, (T * k,))
    rows = T * k if rows is None else rows
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, H // 2), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((rows, H // block), dtype=torch.uint8, device=dev)
    _need(codes, "codes", torch.uint8, (rows, H // 2))
    _need(scales, "scales", torch.uint8, (rows, H // block))
    _check("moe_expand_fp4", load_library().moe_expand_fp4(_ptr(x), T, H, int(k), _ptr(inv_perm), rows, code,
                                                           float(global_scale), _ptr(codes), _ptr(scales),
                                                           _stream_ptr(stream, dev)))
    return codes, scales


# ---------------------------------------------------------------------------
# QK RMSNorm (in place)
# ---------------------------------------------------------------------------

def moe_qk_rmsnorm(q: torch.Tensor, k: torch.Tensor, q_weight: torch.Tensor, k_weight: torch.Tensor,
                   weight_bias: float = 0.0, eps: float = 1e-6, *,
                   stream: Optional[torch.cuda.Stream] = None):
    """Per-head RMSNorm of ``q [T, nq, head_dim]`` and ``k [T, nk, head_dim]``
    (bfloat16) in place: ``(w + weight_bias) * x * rsqrt(mean(x^2) + eps)``.
    Returns ``(q, k)``."""
    T, nq, hd = q.shape
    nk = k.shape[1]
    _need(q, "q", torch.bfloat16, (T, nq, hd))
    _need(k, "k", torch.bfloat16, (T, nk, hd))
    _need(q_weight, "q_weight", torch.bfloat16, (hd,))
    _need(k_weight, "k_weight", torch.bfloat16, (hd,))
    _check("moe_qk_rmsnorm", load_library().moe_qk_rmsnorm(_ptr(q), _ptr(k), T, nq, nk, hd, _ptr(q_weight),
                                                           _ptr(k_weight), float(weight_bias), float(eps),
                                                           _stream_ptr(stream, q.device)))
    return q, k
