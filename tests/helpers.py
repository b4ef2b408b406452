"""Shared test utilities: fixture parsing and the parity checks.

Tolerances
----------
* Integer and byte outputs (top-k ids, counts, offsets, permutation, expanded
  rows): bit-exact.
* bfloat16 outputs of real arithmetic (SwiGLU, combine): elementwise
  ``|gpu - ref| <= ATOL + RTOL * |ref|`` with ATOL = 2e-2, RTOL = 1e-2, where
  ``ref`` is the oracle's once-rounded real result. The kernels compute in
  float32 and round once, so they differ from the exact result by at most one
  bfloat16 unit in the last place (2^-8 relative, about 0.4%) plus a few
  float32 ulps, well inside the bound.
* float32 routing weights: ``|gpu - ref| <= W_ATOL + W_RTOL * |ref|`` with
  W_RTOL = 1e-5, W_ATOL = 1e-7. The kernel's softmax rounds a handful of
  float32 operations per weight (exp, a tree sum over at most 1024 experts =
  10 levels, one division): under 16 roundings of 2^-24 relative each, about
  1e-6, taken with 10x headroom.
"""
from __future__ import annotations

import os

import numpy as np

ATOL = 2e-2
RTOL = 1e-2
W_ATOL = 1e-7
W_RTOL = 1e-5

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name: str) -> dict:
    """Parse a ``key v1 v2 ...`` text fixture (``#`` starts a comment)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def bf16_bits_to_f64(a) -> np.ndarray:
    """bfloat16 bit patterns -> float64 by shifting into a float32 (exact)."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp_distance(a, b) -> np.ndarray:
    """Distance in representable bfloat16 steps between two bit-pattern arrays
    (treating +0 and -0 as the same point)."""
    def ordered(x):
        x = np.asarray(x, dtype=np.uint16).astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def check_bf16_close(got, ref, what: str = "", atol: float = ATOL, rtol: float = RTOL,
                     chunk: int = 1 << 23) -> dict:
    """Assert the elementwise allclose bound on bfloat16 bit patterns; return
    statistics (max abs / rel error, fraction of bit-exact elements, largest
    distance in bfloat16 steps). Large arrays are compared in chunks of
    `chunk` elements, so host memory stays bounded."""
    got = np.asarray(got, dtype=np.uint16)
    ref = np.asarray(ref, dtype=np.uint16)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    gf, rf = got.reshape(-1), ref.reshape(-1)
    n = gf.size
    max_abs = max_rel = 0.0
    exact = 0
    max_ulp = 0
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        gc, rc = gf[lo:hi], rf[lo:hi]
        g = bf16_bits_to_f64(gc)
        r = bf16_bits_to_f64(rc)
        assert np.isfinite(g).all(), f"{what}: non-finite values in the result"
        err = np.abs(g - r)
        bad = err > atol + rtol * np.abs(r)
        if bad.any():
            idx = [np.unravel_index(lo + int(i), got.shape) for i in np.flatnonzero(bad)[:5]]
            raise AssertionError(f"{what}: {int(bad.sum())} elements of [{lo}, {hi}) outside "
                                 f"{atol} + {rtol}*|ref|; first at {[tuple(map(int, i)) for i in idx]}")
        max_abs = max(max_abs, float(err.max()))
        max_rel = max(max_rel, float((err / np.maximum(np.abs(r), 1e-30)).max()))
        exact += int((gc == rc).sum())
        max_ulp = max(max_ulp, int(bf16_ulp_distance(gc, rc).max()))
    return {"max_abs": max_abs, "max_rel": max_rel, "exact_frac": exact / n if n else 1.0,
            "max_ulp": max_ulp}


def check_quant_where_inputs_agree(codes, scales, ref_codes, ref_scales, act, ref_act, block: int,
                                   fp4: bool, what: str = "", min_scale_frac: float = 0.999,
                                   min_code_frac: float = 0.99) -> dict:
    """Block-quantized output of the GPU against the oracle's quantization of
    the oracle's OWN bfloat16 values (no GPU value is fed to the oracle).
    The GPU and the oracle may round a few bfloat16 values of the activation
    differently (both are within the bfloat16 tolerance); everywhere they
    agree, quantization leaves no freedom:
      * a block whose bfloat16 values all agree bit for bit has the oracle's
        scale;
      * an element whose bfloat16 value agrees and whose block scale agrees
        has the oracle's code.
    The scales must agree on at least `min_scale_frac` of the blocks and the
    second rule must cover at least `min_code_frac` of the elements.
    `codes` are one byte per value (MX FP8) or two E2M1 codes per byte with
    element 2i in the low nibble (`fp4`)."""
    act = np.asarray(act, dtype=np.uint16)
    ref_act = np.asarray(ref_act, dtype=np.uint16)
    rows, n = act.shape
    nb = n // block

    def per_elem(c):
        c = np.asarray(c, dtype=np.uint8)
        if not fp4:
            return c
        out = np.empty((c.shape[0], c.shape[1] * 2), dtype=np.uint8)
        out[:, 0::2] = c & 0x0F
        out[:, 1::2] = c >> 4
        return out

    c, rc = per_elem(codes), per_elem(ref_codes)
    s, rs = np.asarray(scales), np.asarray(ref_scales)
    assert c.shape == rc.shape == (rows, n) and s.shape == rs.shape == (rows, nb), what
    same_elem = act == ref_act
    same_blk = same_elem.reshape(rows, nb, block).all(axis=2)
    bad = same_blk & (s != rs)
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} blocks with identical inputs but another scale, "
                             f"first at {np.argwhere(bad)[:5].tolist()}")
    same_scale = s == rs
    mask = same_elem & np.repeat(same_scale, block, axis=1)
    bad = mask & (c != rc)
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} codes differ where value and scale agree, "
                             f"first at {np.argwhere(bad)[:5].tolist()}")
    stats = {"scale_frac": float(same_scale.mean()), "covered_frac": float(mask.mean()),
             "block_same_frac": float(same_blk.mean())}
    assert stats["scale_frac"] >= min_scale_frac, (what, stats)
    assert stats["covered_frac"] >= min_code_frac, (what, stats)
    return stats


def check_weights_close(got, ref, what: str = "topk_weights") -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    bad = err > W_ATOL + W_RTOL * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} weights outside tolerance, first "
                             f"{idx.tolist()}, max err {err.max():.3g}")
    return float(err.max()) if err.size else 0.0


def check_exact(got, ref, what: str = ""):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    if not np.array_equal(got, ref):
        diff = np.argwhere(got != ref)
        raise AssertionError(f"{what}: {len(diff)} mismatches, first at {diff[:5].tolist()}")
