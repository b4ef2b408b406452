"""numpy front end of the plain C oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU-baseline / reference leg, never by the product path. It
shares no code with the CUDA library and imports nothing from it.

Every function mirrors one definition in ``moe_oracle.c`` (see that file for
the page citations and the readings taken where the pages are silent).
bfloat16 arrays are numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmoe_oracle.so`` (plain C, IEEE
    double, no FP contraction so x86 and Arm round alike)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "cc")
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_bf16_round.argtypes = [_f64p, ctypes.c_long, _u16p]
        lib.oracle_bf16_round.restype = None
        lib.oracle_bf16_decode.argtypes = [_u16p, ctypes.c_long, _f64p]
        lib.oracle_bf16_decode.restype = None
        lib.oracle_route_topk.argtypes = [_f32p, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, _i32p, _f32p]
        lib.oracle_route_topk.restype = ctypes.c_int
        lib.oracle_route_permute.argtypes = [_i32p, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                             _i32p, _i32p, _i32p, _i32p]
        lib.oracle_route_permute.restype = ctypes.c_int
        lib.oracle_route_permute_local.argtypes = [_i32p, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_long, _i32p, _i32p, _i32p, _i32p]
        lib.oracle_route_permute_local.restype = ctypes.c_int
        lib.oracle_e4m3_round.argtypes = [_f64p, ctypes.c_long, ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_e4m3_round.restype = None
        lib.oracle_quant_mxfp8.argtypes = [_u16p, ctypes.c_long, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_quant_mxfp8.restype = None
        lib.oracle_e2m1_round.argtypes = [_f64p, ctypes.c_long, ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_e2m1_round.restype = None
        lib.oracle_quant_mxfp4.argtypes = [_u16p, ctypes.c_long, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_quant_mxfp4.restype = None
        lib.oracle_quant_nvfp4.argtypes = [_u16p, ctypes.c_long, ctypes.c_int, ctypes.c_float,
                                           ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint8)]
        lib.oracle_quant_nvfp4.restype = None
        lib.oracle_rmsnorm_heads.argtypes = [_u16p, ctypes.c_long, ctypes.c_int, _u16p, ctypes.c_double,
                                             ctypes.c_double, _u16p]
        lib.oracle_rmsnorm_heads.restype = None
        lib.oracle_expand.argtypes = [_u16p, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                      _i32p, ctypes.c_long, _u16p]
        lib.oracle_expand.restype = ctypes.c_int
        lib.oracle_swiglu.argtypes = [_u16p, ctypes.c_long, ctypes.c_int, _u16p]
        lib.oracle_swiglu.restype = None
        lib.oracle_combine.argtypes = [_u16p, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_long, _f32p, _i32p, _u16p]
        lib.oracle_combine.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# bfloat16 helpers
# --------------------------------------------------------------------------

def bf16_round(v) -> np.ndarray:
    """Round reals (float64) once to bfloat16 bit patterns, nearest-even."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_round(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint16))
    return out


def bf16_decode(h) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_bf16_decode(_ptr(h, ctypes.c_uint16), h.size, _ptr(out, ctypes.c_double))
    return out


# --------------------------------------------------------------------------
# the path
# --------------------------------------------------------------------------

def route_topk(logits, k: int, renorm: bool):
    """Softmax over E, top-k by logit (ties -> lower expert), optional renorm.
    Returns (topk_ids int32 [T,k], topk_weights float32 [T,k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    rc = _load().oracle_route_topk(_ptr(logits, ctypes.c_float), T, E, k, int(bool(renorm)),
                                   _ptr(ids, ctypes.c_int32), _ptr(w, ctypes.c_float))
    if rc != 0:
        raise ValueError("oracle_route_topk: bad sizes")
    return ids, w


def route_permute(topk_ids, E: int):
    """Histogram, exclusive scan and stable counting sort of the flat slots.
    Returns (counts [E], offsets [E+1], perm [S], inv_perm [S]) as int32."""
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    S = T * k
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(S, dtype=np.int32)
    inv_perm = np.empty(S, dtype=np.int32)
    rc = _load().oracle_route_permute(_ptr(ids, ctypes.c_int32), T, E, k,
                                      _ptr(counts, ctypes.c_int32), _ptr(offsets, ctypes.c_int32),
                                      _ptr(perm, ctypes.c_int32), _ptr(inv_perm, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle_route_permute: expert id out of range")
    return counts, offsets, perm, inv_perm


def route(logits, k: int, renorm: bool):
    """Routing as one call: returns a dict with topk_ids, topk_weights,
    expert_counts, expert_offsets, perm, inv_perm."""
    ids, w = route_topk(logits, k, renorm)
    E = np.asarray(logits).shape[1]
    counts, offsets, perm, inv_perm = route_permute(ids, E)
    return {"topk_ids": ids, "topk_weights": w, "expert_counts": counts,
            "expert_offsets": offsets, "perm": perm, "inv_perm": inv_perm}


def local_rows_capacity(T: int, k: int, n_local: int, pad: int) -> int:
    """Rows a padded local buffer may need at most: every slot local, every
    local expert's segment padded by pad - 1."""
    return T * k + n_local * (pad - 1)


def route_permute_local(topk_ids, E: int, e0: int, e1: int, pad: int, rows: int = None):
    """Permutation of the slots whose expert lies in [e0, e1), each local
    expert's segment padded to a multiple of pad. Returns (counts [n],
    offsets [n+1], perm [rows], inv_perm [S]); -1 marks padding rows in perm
    and non-local slots in inv_perm."""
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    n = e1 - e0
    if rows is None:
        rows = local_rows_capacity(T, k, n, pad)
    counts = np.empty(n, dtype=np.int32)
    offsets = np.empty(n + 1, dtype=np.int32)
    perm = np.empty(rows, dtype=np.int32)
    inv_perm = np.empty(T * k, dtype=np.int32)
    rc = _load().oracle_route_permute_local(_ptr(ids, ctypes.c_int32), T, E, k, e0, e1, pad, rows,
                                            _ptr(counts, ctypes.c_int32), _ptr(offsets, ctypes.c_int32),
                                            _ptr(perm, ctypes.c_int32), _ptr(inv_perm, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle_route_permute_local: bad arguments")
    return counts, offsets, perm, inv_perm


def expand_into(x, k: int, perm, out) -> np.ndarray:
    """Like expand(), writing into ``out`` and leaving rows with perm < 0 as
    they are."""
    x = _c(x, np.uint16)
    perm = _c(perm, np.int32)
    T, H = x.shape
    assert out.flags["C_CONTIGUOUS"] and out.dtype == np.uint16 and out.shape == (perm.size, H)
    rc = _load().oracle_expand(_ptr(x, ctypes.c_uint16), T, H, k, _ptr(perm, ctypes.c_int32), perm.size,
                               _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_expand: source token out of range")
    return out


def expand(x, k: int, perm) -> np.ndarray:
    """expanded_x[p] = x[perm[p] // k] for every entry of ``perm`` (bit copy)."""
    x = _c(x, np.uint16)
    perm = _c(perm, np.int32)
    T, H = x.shape
    P = perm.size
    out = np.empty((P, H), dtype=np.uint16)
    rc = _load().oracle_expand(_ptr(x, ctypes.c_uint16), T, H, k, _ptr(perm, ctypes.c_int32), P,
                               _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_expand: source token out of range")
    return out


def swiglu(gate_up) -> np.ndarray:
    """act[r, i] = bf16(silu(gate_up[r, i]) * gate_up[r, I + i])."""
    gu = _c(gate_up, np.uint16)
    rows, two_i = gu.shape
    assert two_i % 2 == 0
    I = two_i // 2
    out = np.empty((rows, I), dtype=np.uint16)
    _load().oracle_swiglu(_ptr(gu, ctypes.c_uint16), rows, I, _ptr(out, ctypes.c_uint16))
    return out


def combine(expert_out, topk_weights, inv_perm) -> np.ndarray:
    """out[t] = bf16(sum_j w[t,j] * expert_out[inv_perm[t*k+j]])."""
    eo = _c(expert_out, np.uint16)
    w = _c(topk_weights, np.float32)
    inv = _c(inv_perm, np.int32).reshape(-1)
    S, H = eo.shape
    T, k = w.shape
    assert inv.size == T * k
    out = np.empty((T, H), dtype=np.uint16)
    rc = _load().oracle_combine(_ptr(eo, ctypes.c_uint16), S, H, k, T, _ptr(w, ctypes.c_float),
                                _ptr(inv, ctypes.c_int32), _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_combine: row index out of range")
    return out


def e4m3_round(v) -> np.ndarray:
    """Round reals to E4M3 bytes (nearest even, saturating to +-448)."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_round(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint8))
    return out


def e4m3_decode(b) -> np.ndarray:
    """E4M3 bytes -> float64 (0x7F/0xFF are NaN). A table written from the
    format's definition (sign, 4-bit exponent with bias 7, 3-bit fraction)."""
    b = np.asarray(b, dtype=np.uint8)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def quant_mxfp8(x_bf16):
    """MXFP8 quantization of a [rows, n] bfloat16 matrix (n % 32 == 0):
    returns (codes uint8 [rows, n], scales uint8 [rows, n/32])."""
    x = _c(x_bf16, np.uint16)
    rows, n = x.shape
    assert n % 32 == 0
    codes = np.empty((rows, n), dtype=np.uint8)
    scales = np.empty((rows, n // 32), dtype=np.uint8)
    _load().oracle_quant_mxfp8(_ptr(x, ctypes.c_uint16), rows, n, _ptr(codes, ctypes.c_uint8),
                               _ptr(scales, ctypes.c_uint8))
    return codes, scales


def dequant_mxfp8(codes, scales) -> np.ndarray:
    """codes * 2^(scale - 127), float64."""
    codes = np.asarray(codes)
    rows, n = codes.shape
    x = np.asarray(scales).astype(np.float64) - 127.0
    return e4m3_decode(codes) * np.repeat(2.0 ** x, 32, axis=1).reshape(rows, n)


def e2m1_round(v) -> np.ndarray:
    """Round reals to E2M1 codes 0..15 (nearest, ties to the even code,
    saturating to +-6, sign kept)."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e2m1_round(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint8))
    return out


def e2m1_decode(c) -> np.ndarray:
    """E2M1 codes (0..15) -> float64, from the format's definition: sign bit
    0x8, exponent bits 0x6 with bias 1, mantissa bit 0x1 (exponent 0 is
    subnormal: 0.m * 2^0)."""
    c = np.asarray(c, dtype=np.uint8)
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = ((c >> 1) & 0x3).astype(np.float64)
    m = (c & 1).astype(np.float64)
    val = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * 2.0 ** (e - 1.0))
    return sign * val


def unpack_fp4(codes) -> np.ndarray:
    """[rows, n/2] bytes -> [rows, n] codes (element 2i in the low nibble)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0x0F
    out[..., 1::2] = codes >> 4
    return out


def quant_mxfp4(x_bf16):
    """MXFP4 of a [rows, n] bfloat16 matrix (n % 32 == 0): returns (codes
    uint8 [rows, n/2], two per byte, scales uint8 [rows, n/32] E8M0)."""
    x = _c(x_bf16, np.uint16)
    rows, n = x.shape
    assert n % 32 == 0
    codes = np.zeros((rows, n // 2), dtype=np.uint8)
    scales = np.empty((rows, n // 32), dtype=np.uint8)
    _load().oracle_quant_mxfp4(_ptr(x, ctypes.c_uint16), rows, n, _ptr(codes, ctypes.c_uint8),
                               _ptr(scales, ctypes.c_uint8))
    return codes, scales


def dequant_mxfp4(codes, scales) -> np.ndarray:
    """E2M1(code) * 2^(scale - 127), float64, [rows, n]."""
    c = unpack_fp4(codes)
    rows, n = c.shape
    x = np.asarray(scales).astype(np.float64) - 127.0
    return e2m1_decode(c) * np.repeat(2.0 ** x, 32, axis=1).reshape(rows, n)


def quant_nvfp4(x_bf16, global_scale: float):
    """NVFP4 of a [rows, n] bfloat16 matrix (n % 16 == 0) with tensor scale
    g > 0: returns (codes uint8 [rows, n/2], scales uint8 [rows, n/16] E4M3)."""
    x = _c(x_bf16, np.uint16)
    rows, n = x.shape
    assert n % 16 == 0
    codes = np.zeros((rows, n // 2), dtype=np.uint8)
    scales = np.empty((rows, n // 16), dtype=np.uint8)
    _load().oracle_quant_nvfp4(_ptr(x, ctypes.c_uint16), rows, n, float(global_scale),
                               _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return codes, scales


def dequant_nvfp4(codes, scales, global_scale: float) -> np.ndarray:
    """E2M1(code) * E4M3(scale) / g, float64, [rows, n]."""
    c = unpack_fp4(codes)
    rows, n = c.shape
    s = e4m3_decode(scales)
    return e2m1_decode(c) * np.repeat(s / float(global_scale), 16, axis=1).reshape(rows, n)


def rmsnorm_heads(x, w, bias: float, eps: float) -> np.ndarray:
    """Per-head RMSNorm: x [..., head_dim] bfloat16 bits, w [head_dim];
    returns bf16((w + bias) * x / sqrt(mean(x^2) + eps))."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    hd = x.shape[-1]
    assert w.shape == (hd,)
    out = np.empty_like(x)
    _load().oracle_rmsnorm_heads(_ptr(x, ctypes.c_uint16), x.size // hd, hd, _ptr(w, ctypes.c_uint16),
                                 float(bias), float(eps), _ptr(out, ctypes.c_uint16))
    return out


def qk_norm(q, k, q_weight, k_weight, bias: float, eps: float):
    """QK norm of q [T, nq, hd] and k [T, nk, hd]: each head normalised with
    its tensor's weight. Returns (q_out, k_out)."""
    return rmsnorm_heads(q, q_weight, bias, eps), rmsnorm_heads(k, k_weight, bias, eps)


def path(logits, x, gate_up, expert_out, k: int, renorm: bool):
    """One pass of the whole path (route, expand, SwiGLU, combine) on host
    arrays. ``gate_up`` and ``expert_out`` stand in for the expert GEMM outputs
    (they are inputs here, as the GEMMs are not part of the path)."""
    r = route(logits, k, renorm)
    r["expanded_x"] = expand(x, k, r["perm"])
    r["act"] = swiglu(gate_up)
    r["out"] = combine(expert_out, r["topk_weights"], r["inv_perm"])
    return r


if __name__ == "__main__":  # pragma: no cover - manual build entry
    print(build(force="--force" in sys.argv))
