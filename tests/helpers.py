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


def check_bf16_close(got, ref, what: str = "", atol: float = ATOL, rtol: float = RTOL) -> dict:
    """Assert the elementwise allclose bound on bfloat16 bit patterns; return
    statistics (max abs / rel error, fraction of bit-exact elements)."""
    got = np.asarray(got, dtype=np.uint16)
    ref = np.asarray(ref, dtype=np.uint16)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    g = bf16_bits_to_f64(got)
    r = bf16_bits_to_f64(ref)
    assert np.isfinite(g).all(), f"{what}: non-finite values in the result"
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    bad = err > bound
    stats = {
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel": float((err / np.maximum(np.abs(r), 1e-30)).max()) if err.size else 0.0,
        "exact_frac": float((got == ref).mean()) if err.size else 1.0,
        "max_ulp": int(bf16_ulp_distance(got, ref).max()) if err.size else 0,
    }
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside "
                             f"{atol} + {rtol}*|ref|; first at {idx.tolist()}; stats {stats}")
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
