"""FP4 outputs (E2M1 codes) of SwiGLU and expand, NVFP4 (E4M3 scale per 16
under a float32 tensor scale) and MXFP4 (E8M0 scale per 32), on the GPU
through the C ABI, against the oracle.

expand_fp4 quantizes bfloat16 input rows, so it must be bit-exact. The fused
swiglu_fp4 quantizes the bfloat16 act it computes in float32, the same values
moe_swiglu stores, so the oracle's quantization of moe_swiglu's output must
match it bit for bit; against the oracle's own (once-rounded) act, codes may
move by one E2M1 step where the act differs by one bfloat16 ulp."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import check_exact, check_quant_where_inputs_agree

pytestmark = pytest.mark.gpu

FORMATS = [("nvfp4", 1.0), ("nvfp4", 448.0 * 6.0 / 40.0), ("nvfp4", 1e-3), ("mxfp4", 0.0)]


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


def _quant(O, fmt, g, x):
    return O.quant_nvfp4(x, g) if fmt == "nvfp4" else O.quant_mxfp4(x)


def _values(O, shape, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(shape) * np.exp(rng.uniform(-6, 6, (shape[0], 1)))
    v[0, :32] = 0.0                                    # all-zero blocks
    v[0, 32:48] = -0.0                                 # negative zeros: codes 0x8
    if shape[0] > 1:
        v[1, 32:64] = 2.0 ** -130                      # subnormal bf16 values
    if shape[0] > 2:
        v[2, :32] = np.linspace(-3e38, 3e38, 32)       # near the top of the bf16 range
    if shape[0] > 3:
        v[3, :16] = [6.0, 5.0, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -6.0, -5.0, -3.5, -2.5, -0.75, -0.25, 0.0, 7.0]
    return O.bf16_round(v)


@pytest.mark.parametrize("fmt,g", FORMATS)
@pytest.mark.parametrize("T,H,E,k", [(64, 256, 8, 2), (4096, 2048, 128, 8), (16, 7168, 256, 8),
                                     (1023, 2880, 32, 4), (9, 48, 8, 3)])
@pytest.mark.parametrize("wide", [True, False])
def test_expand_fp4_bit_exact(dev, oracle_mod, fmt, g, T, H, E, k, wide):
    from memory_bound_moe_gb300 import moe_expand_fp4
    O = oracle_mod
    if fmt == "mxfp4" and H % 32:
        pytest.skip("MXFP4 needs H % 32 == 0")
    logits = np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)
    r = O.route(logits, k, True)
    x = _values(O, (T, H), T + H)
    xd = bf16_dev(x, dev)
    if not wide:
        xd = _offset16(xd)
    codes, scales = moe_expand_fp4(xd, torch.from_numpy(r["inv_perm"]).to(dev), k, fmt, g)
    torch.cuda.synchronize()
    ref_codes, ref_scales = _quant(O, fmt, g, O.expand(x, k, r["perm"]))
    check_exact(scales.cpu().numpy(), ref_scales, f"{fmt} scales T={T} H={H}")
    check_exact(codes.cpu().numpy(), ref_codes, f"{fmt} codes T={T} H={H}")


@pytest.mark.parametrize("fmt,g", [("nvfp4", 2.0), ("mxfp4", 0.0)])
def test_expand_fp4_into_padded_local_rows(dev, oracle_mod, fmt, g):
    from memory_bound_moe_gb300 import moe_expand_fp4, moe_route_local
    O = oracle_mod
    T, H, E, k, e0, e1, pad = 512, 1024, 64, 4, 16, 32, 128
    block = 16 if fmt == "nvfp4" else 32
    logits = np.random.default_rng(1).standard_normal((T, E)).astype(np.float32)
    r = moe_route_local(torch.from_numpy(logits).to(dev), k, True, e0, e1, pad)
    rows = r.perm.numel()
    x = _values(O, (T, H), 9)
    codes = torch.full((rows, H // 2), 0xAB, dtype=torch.uint8, device=dev)
    scales = torch.full((rows, H // block), 0xCD, dtype=torch.uint8, device=dev)
    moe_expand_fp4(bf16_dev(x, dev), r.inv_perm, k, fmt, g, rows, codes=codes, scales=scales)
    torch.cuda.synchronize()
    perm = r.perm.cpu().numpy()
    valid = perm >= 0
    full_c, full_s = _quant(O, fmt, g, x)                  # quantize token rows once
    ref_c = np.full((rows, H // 2), 0xAB, dtype=np.uint8)
    ref_s = np.full((rows, H // block), 0xCD, dtype=np.uint8)
    ref_c[valid] = full_c[perm[valid] // k]
    ref_s[valid] = full_s[perm[valid] // k]
    check_exact(codes.cpu().numpy(), ref_c, f"{fmt} padded codes")
    check_exact(scales.cpu().numpy(), ref_s, f"{fmt} padded scales")


@pytest.mark.parametrize("fmt,g", FORMATS)
@pytest.mark.parametrize("rows,I", [(128, 128), (32768, 768), (128, 2048), (4092, 2880), (7, 32)])
@pytest.mark.parametrize("wide", [True, False])
def test_swiglu_fp4_against_oracle(dev, oracle_mod, fmt, g, rows, I, wide):
    from memory_bound_moe_gb300 import moe_swiglu, moe_swiglu_fp4
    O = oracle_mod
    rng = np.random.default_rng(rows + I)
    gu = O.bf16_round(rng.standard_normal((rows, 2 * I)) * 2)
    gd = bf16_dev(gu, dev)
    if not wide:
        gd = _offset16(gd)
    codes, scales = moe_swiglu_fp4(gd, fmt, g)
    act = moe_swiglu(gd)
    torch.cuda.synchronize()
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    # exact: the oracle's quantization of the GPU's own bfloat16 act
    ec, es = _quant(O, fmt, g, u16(act))
    check_exact(s, es, f"{fmt} scales rows={rows} I={I}")
    check_exact(c, ec, f"{fmt} codes rows={rows} I={I}")
    # near: against the oracle's act, dequantized values within one E2M1 unit
    ref_act = O.swiglu(gu)
    rc, rs = _quant(O, fmt, g, ref_act)
    # independent: the oracle's quantization of its own act, wherever the
    # bfloat16 act and the block scale agree
    check_quant_where_inputs_agree(c, s, rc, rs, u16(act), ref_act, 16 if fmt == "nvfp4" else 32, True,
                                   f"{fmt} rows={rows} I={I}")
    if fmt == "nvfp4":
        deq, ref = O.dequant_nvfp4(c, s, g), O.dequant_nvfp4(rc, rs, g)
        unit = np.repeat(np.maximum(O.e4m3_decode(s), O.e4m3_decode(rs)), 16, axis=1) / g
    else:
        deq, ref = O.dequant_mxfp4(c, s), O.dequant_mxfp4(rc, rs)
        unit = np.repeat(2.0 ** (np.maximum(s, rs).astype(np.float64) - 127), 32, axis=1)
    assert np.all(np.abs(deq - ref) <= 2 * unit * (1 + 1e-6)), fmt
    assert (c == rc).mean() >= 0.99, fmt


def test_fp4_prefill_full(dev, oracle_mod, oracle_act):
    """The prefill shapes in full: SwiGLU 16384 x 14336 outputs (NVFP4 with a
    calibrated tensor scale) and expand of 8192 x 4096 token rows (MXFP4).
    SwiGLU: bit-exact against the oracle's quantization of the GPU's bfloat16
    act, and against the oracle's quantization of its own act wherever the
    two acts and the block scale agree; expand: bit-exact."""
    from memory_bound_moe_gb300 import moe_expand_fp4, moe_swiglu, moe_swiglu_fp4
    from memory_bound_moe_gb300.workloads import WORKLOADS, as_u16, generate
    O = oracle_mod
    w = WORKLOADS["prefill"]
    gu, ref_act = oracle_act("prefill")
    gd = bf16_dev(gu, dev)
    act = moe_swiglu(gd)
    g = 448.0 * 6.0 / float(act.float().abs().max())
    codes, scales = moe_swiglu_fp4(gd, "nvfp4", g)
    torch.cuda.synchronize()
    del gd
    a16, c, s = u16(act), codes.cpu().numpy(), scales.cpu().numpy()
    del act, codes, scales
    rows = a16.shape[0]
    for lo in range(0, rows, 1024):
        hi = min(rows, lo + 1024)
        ec, es = O.quant_nvfp4(a16[lo:hi], g)
        check_exact(s[lo:hi], es, f"prefill swiglu scales [{lo},{hi})")
        check_exact(c[lo:hi], ec, f"prefill swiglu codes [{lo},{hi})")
        rc, rs = O.quant_nvfp4(ref_act[lo:hi], g)
        check_quant_where_inputs_agree(c[lo:hi], s[lo:hi], rc, rs, a16[lo:hi], ref_act[lo:hi], 16, True,
                                       f"prefill swiglu [{lo},{hi})")
    x = as_u16(generate(w, seed=0, parts=("x",))["x"])
    T, k = w.T, w.k
    inv = torch.arange(T * k, dtype=torch.int32, device=dev)        # identity rows: row t*k+j = token t
    codes, scales = moe_expand_fp4(bf16_dev(x, dev), inv, k, "mxfp4")
    torch.cuda.synchronize()
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    ec, es = O.quant_mxfp4(x)
    for j in range(k):
        check_exact(s[j::k], es, f"prefill expand scales j={j}")
        check_exact(c[j::k], ec, f"prefill expand codes j={j}")
