"""The row expansion's two unroll depths.

moe_expand gives every warp one item (a token and a chunk of 32*U vectors of
its row) at a time: U = 2 once the batch has enough such items to fill every
SM a few times over, U = 1 below that. The default library runs the small
shapes of the parity tests with U = 1 and the large workloads with U = 2; a
second copy of the library is built with the threshold at 0, so that every
shape below runs with U = 2, including rows that end inside a chunk, both
vector widths, and padded local rows whose -1 entries are skipped. Each must
be bit-exact against the oracle.
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
    L = ctypes.CDLL(build.build(defines=["MOE_EXPAND_U2_MIN_WARPS_PER_SM=0"],
                                out_dir=os.path.join(pkg, "lib", "expand_u2")))
    L.moe_expand.argtypes = [_vp, _i64, _i32, _i32, _vp, _vp, _vp]
    L.moe_expand_rows.argtypes = [_vp, _i64, _i32, _i32, _vp, _i64, _vp, _vp]
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
