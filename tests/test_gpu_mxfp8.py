"""MXFP8 outputs (E4M3 codes, E8M0 scale per 32) of SwiGLU and expand, on the
GPU through the C ABI, against the oracle.

expand_mxfp8 quantizes bfloat16 input rows, so it must be bit-exact.
swiglu_mxfp8 quantizes the bfloat16 act the kernel computes in float32; where
that act differs from the oracle's once-rounded act by one bfloat16 ulp the
quantized code can differ by one E4M3 step, so the bar is: scales equal in
every block (allowing 1 in 10^4 blocks where the block maximum straddles a
power of two), dequantized values within one E4M3 spacing of the oracle's
(2^-3 relative for normals, 2^(X-9) absolute for subnormals), and at least
99.9% of codes equal."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import check_exact, check_quant_where_inputs_agree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_moe_gb300 import build
    build.build()
    return torch.device("cuda:0")


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


def _values(O, shape, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(shape) * np.exp(rng.uniform(-6, 6, (shape[0], 1)))
    v[0, :32] = 0.0                                    # an all-zero block
    if shape[0] > 1:
        v[1, 32:64] = 2.0 ** -130                      # subnormal bf16 block
    if shape[0] > 2:
        v[2, :32] = np.linspace(-3e38, 3e38, 32)       # near the top of the bf16 range
    return O.bf16_round(v)


@pytest.mark.parametrize("T,H,E,k", [(64, 256, 8, 2), (4096, 2048, 128, 8), (16, 7168, 256, 8),
                                     (1023, 2880, 32, 4), (8192, 4096, 8, 2)])
@pytest.mark.parametrize("wide", [True, False])
def test_expand_mxfp8_bit_exact(dev, oracle_mod, T, H, E, k, wide):
    from memory_bound_moe_gb300 import moe_expand_mxfp8
    O = oracle_mod
    logits = np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)
    r = O.route(logits, k, True)
    x = _values(O, (T, H), T + H)
    xd = bf16_dev(x, dev)
    if not wide:
        xd = _offset16(xd)
    codes, scales = moe_expand_mxfp8(xd, torch.from_numpy(r["inv_perm"]).to(dev), k)
    torch.cuda.synchronize()
    ref_codes, ref_scales = O.quant_mxfp8(O.expand(x, k, r["perm"]))
    check_exact(scales.cpu().numpy(), ref_scales, f"scales T={T} H={H}")
    check_exact(codes.cpu().numpy(), ref_codes, f"codes T={T} H={H}")


def test_expand_mxfp8_into_padded_local_rows(dev, oracle_mod):
    from memory_bound_moe_gb300 import moe_expand_mxfp8, moe_route_local
    O = oracle_mod
    T, H, E, k, e0, e1, pad = 512, 1024, 64, 4, 16, 32, 128
    logits = np.random.default_rng(1).standard_normal((T, E)).astype(np.float32)
    r = moe_route_local(torch.from_numpy(logits).to(dev), k, True, e0, e1, pad)
    rows = r.perm.numel()
    x = _values(O, (T, H), 9)
    codes = torch.full((rows, H), 0xAB, dtype=torch.uint8, device=dev)
    scales = torch.full((rows, H // 32), 0xCD, dtype=torch.uint8, device=dev)
    moe_expand_mxfp8(bf16_dev(x, dev), r.inv_perm, k, rows, codes=codes, scales=scales)
    torch.cuda.synchronize()
    perm = r.perm.cpu().numpy()
    valid = perm >= 0
    full_c, full_s = O.quant_mxfp8(x)                       # quantize token rows once
    ref_c = np.full((rows, H), 0xAB, dtype=np.uint8)
    ref_s = np.full((rows, H // 32), 0xCD, dtype=np.uint8)
    ref_c[valid] = full_c[perm[valid] // k]
    ref_s[valid] = full_s[perm[valid] // k]
    check_exact(codes.cpu().numpy(), ref_c, "padded codes")
    check_exact(scales.cpu().numpy(), ref_s, "padded scales")


def _check_swiglu_q(O, codes, scales, gu, what, ref_act=None):
    ref_c, ref_s = O.quant_mxfp8(O.swiglu(gu) if ref_act is None else ref_act)
    same_scale = scales == ref_s
    assert same_scale.mean() >= 1 - 1e-4, (what, float(same_scale.mean()))
    deq = O.dequant_mxfp8(codes, scales)
    ref = O.dequant_mxfp8(ref_c, ref_s)
    X = np.repeat(ref_s.astype(np.float64) - 127, 32, axis=1)
    blk = np.repeat(same_scale, 32, axis=1)
    bound = np.maximum(2.0 ** -3 * np.abs(ref), 2.0 ** (X - 9))
    bad = (np.abs(deq - ref) > bound) & blk
    assert not bad.any(), (what, np.argwhere(bad)[:5])
    assert (codes == ref_c)[blk].mean() >= 0.999, what
    return ref_c, ref_s


@pytest.mark.parametrize("rows,I", [(128, 128), (32768, 768), (128, 2048), (4092, 2880), (7, 32)])
@pytest.mark.parametrize("wide", [True, False])
def test_swiglu_mxfp8_against_oracle(dev, oracle_mod, rows, I, wide):
    from memory_bound_moe_gb300 import moe_swiglu, moe_swiglu_mxfp8
    O = oracle_mod
    rng = np.random.default_rng(rows + I)
    gu = O.bf16_round(rng.standard_normal((rows, 2 * I)) * 2)
    gd = bf16_dev(gu, dev)
    if not wide:
        gd = _offset16(gd)
    codes, scales = moe_swiglu_mxfp8(gd)
    act = u16(moe_swiglu(gd))
    torch.cuda.synchronize()
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    ref_act = O.swiglu(gu)
    ref_c, ref_s = _check_swiglu_q(O, c, s, gu, f"rows={rows} I={I}", ref_act)
    check_quant_where_inputs_agree(c, s, ref_c, ref_s, act, ref_act, 32, False, f"rows={rows} I={I}")


def test_swiglu_mxfp8_prefill_full(dev, oracle_mod, oracle_act):
    """The prefill shape (16384 x 14336 outputs), every block, compared in
    row chunks against the oracle's quantization of its own act."""
    from memory_bound_moe_gb300 import moe_swiglu, moe_swiglu_mxfp8
    O = oracle_mod
    gu, ref_act = oracle_act("prefill")
    gd = bf16_dev(gu, dev)
    codes, scales = moe_swiglu_mxfp8(gd)
    act = u16(moe_swiglu(gd))
    torch.cuda.synchronize()
    del gd
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    rows = gu.shape[0]
    for a in range(0, rows, 1024):
        b = min(rows, a + 1024)
        ref_c, ref_s = _check_swiglu_q(O, c[a:b], s[a:b], None, f"prefill rows {a}:{b}", ref_act[a:b])
        check_quant_where_inputs_agree(c[a:b], s[a:b], ref_c, ref_s, act[a:b], ref_act[a:b], 32, False,
                                       f"prefill rows {a}:{b}")


def test_swiglu_mxfp8_dequantizes_to_swiglu(dev, oracle_mod):
    """GPU self-consistency: the quantized act is the GPU's own bf16 act
    rounded to E4M3 with the block's scale (within half an E4M3 step)."""
    from memory_bound_moe_gb300 import moe_swiglu, moe_swiglu_mxfp8
    O = oracle_mod
    rng = np.random.default_rng(5)
    gu = bf16_dev(O.bf16_round(rng.standard_normal((2048, 2 * 768)) * 3), dev)
    act = O.bf16_decode(u16(moe_swiglu(gu)))
    codes, scales = moe_swiglu_mxfp8(gu)
    torch.cuda.synchronize()
    s = scales.cpu().numpy()
    deq = O.dequant_mxfp8(codes.cpu().numpy(), s)
    X = np.repeat(s.astype(np.float64) - 127, 32, axis=1)
    amax = np.abs(act).reshape(2048, -1, 32).max(axis=2)
    nz = amax > 0
    assert np.array_equal((np.floor(np.log2(amax[nz])) - 8 + 127).astype(int), s[nz].astype(int))
    inside = np.abs(act) / 2.0 ** X <= 448
    bound = np.maximum(2.0 ** -4 * np.abs(act), 2.0 ** (X - 10))
    assert np.all(np.abs(deq - act)[inside] <= bound[inside])
