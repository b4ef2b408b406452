"""The row kernels split jobs of more than 2^30 work items into several
launches over row ranges (so 32-bit grid-stride indices never wrap). Inputs
that large take tens of GB, so this builds a second copy of the library with
the split threshold lowered to 1000 items and runs small inputs through it:
every launcher then issues 5 to 40 launches, each with its own row offset,
and the results must still match the oracle (and the default library)."""
from __future__ import annotations

import ctypes
import os

import numpy as np
import pytest
import torch

from helpers import check_bf16_close, check_exact

pytestmark = pytest.mark.gpu

SPLIT = 1000   # items per launch in the test build


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib(dev):
    from memory_bound_moe_gb300 import build
    pkg = os.path.dirname(build.__file__)
    path = build.build(defines=[f"MOE_MAX_ITEMS_PER_LAUNCH={SPLIT}"],
                       out_dir=os.path.join(pkg, "lib", "split_launch"))
    L = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    L.moe_expand.argtypes = [vp, i64, i32, i32, vp, vp, vp]
    L.moe_swiglu.argtypes = [vp, i64, i32, vp, vp]
    L.moe_combine.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp]
    L.moe_swiglu_mxfp8.argtypes = [vp, i64, i32, vp, vp, vp]
    L.moe_expand_fp4.argtypes = [vp, i64, i32, i32, vp, i64, i32, f32, vp, vp, vp]
    L.moe_qk_rmsnorm.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, f32, f32, vp]
    return L


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _stream(dev):
    return torch.cuda.current_stream(dev).cuda_stream


def test_expand_and_combine_split(dev, lib, oracle_mod):
    O = oracle_mod
    T, H, E, k = 100, 2048, 64, 8              # 128 vectors per token: 7 tokens per launch
    rng = np.random.default_rng(0)
    r = O.route(rng.standard_normal((T, E)).astype(np.float32), k, True)
    x = O.bf16_round(rng.standard_normal((T, H)))
    inv = torch.from_numpy(r["inv_perm"]).to(dev)
    ex = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    assert lib.moe_expand(bf16_dev(x, dev).data_ptr(), T, H, k, inv.data_ptr(), ex.data_ptr(), _stream(dev)) == 0
    eo = O.bf16_round(rng.standard_normal((T * k, H)))
    w = torch.from_numpy(r["topk_weights"]).to(dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    assert lib.moe_combine(bf16_dev(eo, dev).data_ptr(), T, H, k, w.data_ptr(), inv.data_ptr(), out.data_ptr(),
                           _stream(dev)) == 0
    torch.cuda.synchronize()
    check_exact(u16(ex), O.expand(x, k, r["perm"]), "split expand")
    check_bf16_close(u16(out), O.combine(eo, r["topk_weights"], r["inv_perm"]), "split combine")


def test_swiglu_split(dev, lib, oracle_mod):
    O = oracle_mod
    rows, I = 300, 768                         # 48 vectors per row: 20 rows per launch
    gu = O.bf16_round(np.random.default_rng(1).standard_normal((rows, 2 * I)) * 2)
    act = torch.empty((rows, I), dtype=torch.bfloat16, device=dev)
    assert lib.moe_swiglu(bf16_dev(gu, dev).data_ptr(), rows, I, act.data_ptr(), _stream(dev)) == 0
    torch.cuda.synchronize()
    check_bf16_close(u16(act), O.swiglu(gu), "split swiglu")


def test_block_quant_split_matches_default_library(dev, lib, oracle_mod):
    from memory_bound_moe_gb300 import moe_expand_fp4, moe_swiglu_mxfp8
    O = oracle_mod
    rows, I = 200, 768                         # 48 items of 16 values per row: 20 rows per launch
    gu = bf16_dev(O.bf16_round(np.random.default_rng(2).standard_normal((rows, 2 * I)) * 2), dev)
    codes = torch.empty((rows, I), dtype=torch.uint8, device=dev)
    scales = torch.empty((rows, I // 32), dtype=torch.uint8, device=dev)
    assert lib.moe_swiglu_mxfp8(gu.data_ptr(), rows, I, codes.data_ptr(), scales.data_ptr(), _stream(dev)) == 0
    rc, rs = moe_swiglu_mxfp8(gu)
    T, H, E, k = 90, 1024, 32, 4               # 64 items per token: 15 tokens per launch
    r = O.route(np.random.default_rng(3).standard_normal((T, E)).astype(np.float32), k, True)
    x = O.bf16_round(np.random.default_rng(4).standard_normal((T, H)))
    inv = torch.from_numpy(r["inv_perm"]).to(dev)
    c4 = torch.empty((T * k, H // 2), dtype=torch.uint8, device=dev)
    s4 = torch.empty((T * k, H // 16), dtype=torch.uint8, device=dev)
    assert lib.moe_expand_fp4(bf16_dev(x, dev).data_ptr(), T, H, k, inv.data_ptr(), T * k, 0, 3.0,
                              c4.data_ptr(), s4.data_ptr(), _stream(dev)) == 0
    torch.cuda.synchronize()
    assert torch.equal(codes, rc) and torch.equal(scales, rs)
    ec, es = O.quant_nvfp4(O.expand(x, k, r["perm"]), 3.0)
    check_exact(c4.cpu().numpy(), ec, "split expand nvfp4 codes")
    check_exact(s4.cpu().numpy(), es, "split expand nvfp4 scales")


def test_qk_rmsnorm_split(dev, lib, oracle_mod):
    O = oracle_mod
    T, nq, nk, hd = 100, 32, 4, 128            # 36 heads per token: 27 tokens per launch
    rng = np.random.default_rng(5)
    q = O.bf16_round(rng.standard_normal((T, nq, hd)))
    kk = O.bf16_round(rng.standard_normal((T, nk, hd)) * 3)
    qw = O.bf16_round(rng.standard_normal(hd) * 0.2)
    kw = O.bf16_round(rng.standard_normal(hd) * 0.2)
    qd, kd = bf16_dev(q, dev), bf16_dev(kk, dev)
    assert lib.moe_qk_rmsnorm(qd.data_ptr(), kd.data_ptr(), T, nq, nk, hd, bf16_dev(qw, dev).data_ptr(),
                              bf16_dev(kw, dev).data_ptr(), 0.5, 1e-6, _stream(dev)) == 0
    torch.cuda.synchronize()
    rq, rk = O.qk_norm(q, kk, qw, kw, 0.5, 1e-6)
    check_bf16_close(u16(qd), rq, "split q")
    check_bf16_close(u16(kd), rk, "split k")
