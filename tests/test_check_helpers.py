"""The parity checks themselves, on the CPU: the chunked bfloat16 comparison
and the block-quantization check against the oracle's own values must pass
on agreeing data and fail on a planted mistake (a changed element, code or
scale), so that a GPU test built on them cannot pass vacuously."""
from __future__ import annotations

import numpy as np
import pytest

from helpers import check_bf16_close, check_quant_where_inputs_agree


def _bf16(O, v):
    return O.bf16_round(np.asarray(v, dtype=np.float64))


def test_chunked_bf16_check_matches_one_pass_and_finds_the_last_chunk(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(0)
    ref = _bf16(O, rng.standard_normal((37, 64)))
    got = ref.copy()
    got[5, 7] ^= 1                                   # one bfloat16 step off: inside the bound
    one = check_bf16_close(got, ref, "one pass")
    small = check_bf16_close(got, ref, "chunks", chunk=100)
    assert one == small and one["max_ulp"] == 1 and one["exact_frac"] == 1 - 1 / got.size
    bad = got.copy()
    bad[36, 63] = _bf16(O, O.bf16_decode(ref[36:37, 63]) + 1.0)[0]   # far outside, in the last chunk
    with pytest.raises(AssertionError):
        check_bf16_close(bad, ref, "planted", chunk=100)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
def test_quant_agreement_check(oracle_mod, fmt):
    O = oracle_mod
    rng = np.random.default_rng(1)
    rows, n = 64, 256
    ref_act = _bf16(O, rng.standard_normal((rows, n)) * 3)
    # a stand-in for the GPU: the same act with a few values one bfloat16
    # step away, quantized by the oracle
    act = ref_act.copy()
    flip = rng.choice(rows * n, size=20, replace=False)
    act.reshape(-1)[flip] ^= 1
    quant = {"mxfp8": O.quant_mxfp8, "mxfp4": O.quant_mxfp4,
             "nvfp4": lambda a: O.quant_nvfp4(a, 448.0 * 6.0 / 12.0)}[fmt]
    block, fp4 = {"mxfp8": (32, False), "mxfp4": (32, True), "nvfp4": (16, True)}[fmt]
    c, s = quant(act)
    rc, rs = quant(ref_act)
    stats = check_quant_where_inputs_agree(c, s, rc, rs, act, ref_act, block, fp4, fmt)
    assert stats["covered_frac"] > 0.99

    same = (act == ref_act).reshape(-1)
    e = int(np.flatnonzero(same)[3])                  # an element whose value agrees
    r, col = divmod(e, n)
    bad_c = c.copy()
    if fp4:
        bad_c[r, col // 2] ^= 0x01 if col % 2 == 0 else 0x10
    else:
        bad_c[r, col] ^= 0x01
    with pytest.raises(AssertionError):
        check_quant_where_inputs_agree(bad_c, s, rc, rs, act, ref_act, block, fp4, fmt)

    blk_same = (act == ref_act).reshape(rows, n // block, block).all(axis=2)
    br, bb = np.argwhere(blk_same)[0]
    bad_s = s.copy()
    bad_s[br, bb] ^= 0x01
    with pytest.raises(AssertionError):
        check_quant_where_inputs_agree(c, bad_s, rc, rs, act, ref_act, block, fp4, fmt)
