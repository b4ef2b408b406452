"""The row expansion's lane widths, plain and block-quantized.

moe_expand gives every warp one item (a token and a chunk of 32*U vectors of
its row) at a time: U = 2 once the batch has enough such items to fill every
SM a few times over, U = 1 below that. The quantized expansions
(moe_expand_mxfp8, moe_expand_fp4) take the same form with 1 or 2 input
vectors per lane: 2 where whole lane vectors fit the row and the code and
scale buffers are aligned for the wider stores, again once the batch has
enough items. The default library runs the small shapes of the parity tests
with the narrow forms; a second copy of the library is built with both item
thresholds at 0, so that every shape below runs with the widest form its row
length and buffers allow: rows that end inside a chunk, both input vector
widths, code and scale buffers aligned to less than the widest stores, and
padded local rows whose -1 entries are skipped. Each must be bit-exact
against the oracle.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import pytest
import torch

from helpers import check_exact

pytestmark = pytest.mark.gpu

_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def u2_lib(dev):
    from memory_bound_moe_gb300 import build
    pkg = os.path.dirname(build.__file__)
    L = ctypes.CDLL(build.build(defines=["MOE_EXPAND_U2_MIN_WARPS_PER_SM=0", "MOE_EXPAND_Q_MIN_WARPS_PER_SM=0"],
                                out_dir=os.path.join(pkg, "lib", "expand_u2")))
    L.moe_expand.argtypes = [_vp, _i64, _i32, _i32, _vp, _vp, _vp]
    L.moe_expand_rows.argtypes = [_vp, _i64, _i32, _i32, _vp, _i64, _vp, _vp]
    L.moe_expand_mxfp8.argtypes = [_vp, _i64, _i32, _i32, _vp, _i64, _vp, _vp, _vp]
    L.moe_expand_fp4.argtypes = [_vp, _i64, _i32, _i32, _vp, _i64, _i32, ctypes.c_float, _vp, _vp, _vp]
    return L


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _offset16(t):
    flat = torch.empty(t.numel() + 16, dtype=t.dtype, device=t.device)
    shift = ((16 - flat.data_ptr() % 32) % 32) // t.element_size()
    v = flat[shift:shift + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


def _inputs(O, T, H, k, seed):
    rng = np.random.default_rng(seed)
    E = max(k, 8)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    r = O.route(logits, k, True)
    x = O.bf16_round(rng.standard_normal((T, H)))
    return r, x


# T, H, k: one-vector rows up to rows of many chunks, rows ending inside a
# chunk (H = 24, 264, 2880, 4104), k = 1 .. 16
SHAPES = [(1, 8, 1), (3, 16, 2), (17, 24, 3), (100, 264, 5), (33, 2880, 4), (9, 7168, 8), (5, 512, 16),
          (2000, 1024, 2), (1023, 2880, 4), (4096, 2048, 8), (513, 4104, 3), (300, 65536, 2)]


@pytest.mark.parametrize("T,H,k", SHAPES)
@pytest.mark.parametrize("wide", [True, False])
def test_two_vectors_per_lane_match_oracle(dev, u2_lib, oracle_mod, T, H, k, wide):
    O = oracle_mod
    r, x = _inputs(O, T, H, k, seed=T + H + k)
    xd = bf16_dev(x, dev)
    out = torch.full((T * k, H), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
    if not wide:
        xd, out = _offset16(xd), _offset16(out)
    inv = torch.from_numpy(r["inv_perm"]).to(dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    assert u2_lib.moe_expand(xd.data_ptr(), T, H, k, inv.data_ptr(), out.data_ptr(), sp) == 0
    torch.cuda.synchronize(dev)
    check_exact(u16(out), O.expand(x, k, r["perm"]), f"T={T} H={H} k={k}")


def test_two_vectors_per_lane_padded_local_rows(dev, u2_lib, oracle_mod):
    """Padded local rows: inv_perm entries of slots on other ranks are -1 and
    padding rows are never written (their canary stays)."""
    from memory_bound_moe_gb300 import moe_route_local
    O = oracle_mod
    T, H, E, k, e0, e1, pad = 1500, 1024, 64, 4, 16, 40, 128
    logits = np.random.default_rng(3).standard_normal((T, E)).astype(np.float32)
    r = moe_route_local(torch.from_numpy(logits).to(dev), k, True, e0, e1, pad)
    rows = r.perm.numel()
    x = O.bf16_round(np.random.default_rng(4).standard_normal((T, H)))
    out = torch.full((rows, H), 0x5a5a, dtype=torch.int16, device=dev).view(torch.bfloat16)
    sp = torch.cuda.current_stream(dev).cuda_stream
    assert u2_lib.moe_expand_rows(bf16_dev(x, dev).data_ptr(), T, H, k, r.inv_perm.data_ptr(), rows,
                                  out.data_ptr(), sp) == 0
    torch.cuda.synchronize(dev)
    perm = r.perm.cpu().numpy()
    ref = np.full((rows, H), 0x5a5a, dtype=np.uint16)
    O.expand_into(x, k, perm, ref)
    check_exact(u16(out), ref, "padded local rows")


# ---------------------------------------------------------------------------
# Block-quantized expansion

FMT_BLOCK = {"nvfp4": 16, "mxfp4": 32, "mxfp8": 32}
FMT_BITS = {"nvfp4": 4, "mxfp4": 4, "mxfp8": 8}
Q_FORMATS = [("nvfp4", 1.0), ("nvfp4", 448.0 * 6.0 / 40.0), ("mxfp4", 0.0), ("mxfp8", 0.0)]

# T, H, k: rows that take one vector per lane only (16, 48), rows of whole
# chunks (96 .. 7168), rows ending inside a chunk of two-vector lanes (2880,
# 4160), one chunk with idle lanes (512), long rows (65536), k = 1 .. 16
Q_SHAPES = [(3, 16, 2), (17, 48, 3), (9, 96, 5), (40, 160, 1), (33, 2880, 4), (9, 7168, 8), (5, 512, 16),
            (2000, 1024, 2), (513, 4160, 3), (300, 65536, 2)]

# where each buffer starts: "aligned" (x and codes on 32 bytes, scales on
# 4); "x16": x 16 bytes past a 32-byte boundary (16-byte loads);
# "codes16": codes 16 bytes past one (narrower code stores); "scales1":
# scales on an odd address (one scale byte per store)
PLACEMENTS = ["aligned", "x16", "codes16", "scales1"]


def _u8_at(n, mod32, dev, fill):
    """n bytes whose first byte sits mod32 bytes past a 32-byte boundary."""
    flat = torch.full((n + 64,), fill, dtype=torch.uint8, device=dev)
    shift = (mod32 - flat.data_ptr() % 32) % 32
    v = flat[shift:shift + n]
    assert v.data_ptr() % 32 == mod32
    return v


def _quant_ref(O, fmt, g, rows):
    if fmt == "nvfp4":
        return O.quant_nvfp4(rows, g)
    if fmt == "mxfp4":
        return O.quant_mxfp4(rows)
    return O.quant_mxfp8(rows)


def _q_values(O, T, H, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((T, H)) * np.exp(rng.uniform(-6, 6, (T, 1)))
    v[0, :16] = 0.0                                    # an all-zero block
    if T > 1:
        v[1, :16] = [6.0, 5.0, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -6.0, -5.0, -3.5, -2.5, -0.75, -0.25, -0.0, 7.0]
    return O.bf16_round(v)


def _expand_q(lib, fmt, g, xd, T, H, k, inv, rows, codes, scales, sp):
    if fmt == "mxfp8":
        return lib.moe_expand_mxfp8(xd.data_ptr(), T, H, k, inv.data_ptr(), rows, codes.data_ptr(),
                                    scales.data_ptr(), sp)
    return lib.moe_expand_fp4(xd.data_ptr(), T, H, k, inv.data_ptr(), rows, 0 if fmt == "nvfp4" else 1, g,
                              codes.data_ptr(), scales.data_ptr(), sp)


@pytest.mark.parametrize("fmt,g", Q_FORMATS)
@pytest.mark.parametrize("T,H,k", Q_SHAPES)
@pytest.mark.parametrize("place", PLACEMENTS)
def test_quantized_lane_widths_match_oracle(dev, u2_lib, oracle_mod, fmt, g, T, H, k, place):
    O = oracle_mod
    block, bits = FMT_BLOCK[fmt], FMT_BITS[fmt]
    if H % block:
        pytest.skip(f"{fmt} needs H % {block} == 0")
    r, _ = _inputs(O, T, 8, k, seed=T + H + k)
    x = _q_values(O, T, H, seed=T * H + k)
    xd = bf16_dev(x, dev)
    if place == "x16":
        xd = _offset16(xd)
    S = T * k
    cb, sb = S * H * bits // 8, S * H // block
    codes = _u8_at(cb, 16 if place == "codes16" else 0, dev, 0xAB)
    scales = _u8_at(sb, 1 if place == "scales1" else 0, dev, 0xCD)
    inv = torch.from_numpy(r["inv_perm"]).to(dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    assert _expand_q(u2_lib, fmt, g, xd, T, H, k, inv, S, codes, scales, sp) == 0
    torch.cuda.synchronize(dev)
    ref_c, ref_s = _quant_ref(O, fmt, g, O.expand(x, k, r["perm"]))
    check_exact(scales.cpu().numpy().reshape(S, H // block), ref_s, f"{fmt} scales T={T} H={H} k={k} {place}")
    check_exact(codes.cpu().numpy().reshape(S, H * bits // 8), ref_c, f"{fmt} codes T={T} H={H} k={k} {place}")


@pytest.mark.parametrize("fmt,g", Q_FORMATS)
def test_quantized_lane_widths_padded_local_rows(dev, u2_lib, oracle_mod, fmt, g):
    """Padded local rows in the widest quantized form: slots on other ranks
    (-1) and padding rows are never written (their canaries stay)."""
    from memory_bound_moe_gb300 import moe_route_local
    O = oracle_mod
    T, H, E, k, e0, e1, pad = 1500, 1024, 64, 4, 16, 40, 128
    block, bits = FMT_BLOCK[fmt], FMT_BITS[fmt]
    logits = np.random.default_rng(5).standard_normal((T, E)).astype(np.float32)
    r = moe_route_local(torch.from_numpy(logits).to(dev), k, True, e0, e1, pad)
    rows = r.perm.numel()
    x = _q_values(O, T, H, seed=6)
    codes = torch.full((rows, H * bits // 8), 0xAB, dtype=torch.uint8, device=dev)
    scales = torch.full((rows, H // block), 0xCD, dtype=torch.uint8, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    assert _expand_q(u2_lib, fmt, g, bf16_dev(x, dev), T, H, k, r.inv_perm, rows, codes, scales, sp) == 0
    torch.cuda.synchronize(dev)
    perm = r.perm.cpu().numpy()
    valid = perm >= 0
    full_c, full_s = _quant_ref(O, fmt, g, x)          # each token row quantized once
    ref_c = np.full((rows, H * bits // 8), 0xAB, dtype=np.uint8)
    ref_s = np.full((rows, H // block), 0xCD, dtype=np.uint8)
    ref_c[valid] = full_c[perm[valid] // k]
    ref_s[valid] = full_s[perm[valid] // k]
    check_exact(codes.cpu().numpy(), ref_c, f"{fmt} padded codes")
    check_exact(scales.cpu().numpy(), ref_s, f"{fmt} padded scales")
