"""Pins for the CPU oracle: every check here comes from somewhere other than
the oracle itself (closed forms, textbook special cases, library routines of
numpy / PyTorch, brute force, a hand-worked example), chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, swapped
gate/up halves, perm confused with inv_perm, a double rounding) fails one of
them. CPU only.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch

from helpers import bf16_bits_to_f64, bf16_ulp_distance, read_fixture


def _torch_bf16_bits(vals_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(vals_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# bfloat16 rounding and decoding
# ---------------------------------------------------------------------------

def test_bf16_round_known_patterns(oracle_mod):
    o = oracle_mod
    # (value, expected bit pattern); a list, since 0.0 and -0.0 are equal keys
    cases = [
        (1.0, 0x3F80),
        (-2.0, 0xC000),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (1 + 2 ** -8, 0x3F80),            # exact tie -> even (down)
        (1 + 3 * 2 ** -8, 0x3F82),        # exact tie -> even (up)
        (1 + 2 ** -8 + 2 ** -40, 0x3F81),  # just above the tie: one rounding, not two
        (2.0 ** -133, 0x0001),            # smallest subnormal
        (2.0 ** -134, 0x0000),            # half of it: tie -> even zero
        (3 * 2.0 ** -134, 0x0002),        # 1.5 units: tie -> even (2 units)
        ((2 - 2 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
        ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80),   # overflow tie rounds to infinity
        ((2 - 2 ** -8 - 2 ** -20) * 2.0 ** 127, 0x7F7F),
        (math.inf, 0x7F80),
        (-math.inf, 0xFF80),
    ]
    got = o.bf16_round(np.array([v for v, _ in cases], dtype=np.float64))
    assert [int(g) for g in got] == [b for _, b in cases]
    nan = o.bf16_round(np.array([math.nan]))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x007F) != 0


def test_bf16_round_matches_torch_on_float32_values(oracle_mod):
    # A float32 value rounds once to bfloat16 whether it is read as float or
    # double, so torch's float32->bfloat16 conversion is an independent check.
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    normal = rng.standard_normal(50_000).astype(np.float32) * 3
    vals = np.concatenate([vals, normal])
    ours = oracle_mod.bf16_round(vals.astype(np.float64))
    ref = _torch_bf16_bits(vals)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_decode_all_patterns(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.bf16_decode(pats)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


# ---------------------------------------------------------------------------
# routing: top-k
# ---------------------------------------------------------------------------

def _topk_by_sort(row, k):
    # brute force: sort every expert by (logit descending, index ascending)
    return sorted(range(len(row)), key=lambda e: (-float(row[e]), e))[:k]


@pytest.mark.parametrize("E,k", [(2, 1), (4, 2), (8, 2), (8, 8), (12, 5), (33, 4), (130, 8)])
@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_topk_brute_force_sort(oracle_mod, E, k, kind):
    rng = np.random.default_rng(E * 100 + k)
    T = 50
    if kind == "ties":
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
        logits[rng.random((T, E)) < 0.2] = -0.0
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle_mod.route_topk(logits, k, renorm=False)
    for t in range(T):
        assert list(ids[t]) == _topk_by_sort(logits[t], k), (t, logits[t])


@pytest.mark.parametrize("E,k", [(3, 2), (5, 2), (6, 3), (8, 4)])
def test_topk_pairwise_dominance_all_subsets(oracle_mod, E, k):
    # Characterise the selection without sorting: among all C(E, k) subsets,
    # exactly one has every member beating every non-member (larger logit, or
    # equal logit and lower index). The oracle must return that subset, in
    # order of the same relation.
    rng = np.random.default_rng(7 + E)
    logits = rng.integers(-1, 2, size=(40, E)).astype(np.float32)

    def beats(row, a, b):
        return row[a] > row[b] or (row[a] == row[b] and a < b)

    ids, _ = oracle_mod.route_topk(logits, k, renorm=False)
    for t, row in enumerate(logits):
        winners = [set(c) for c in itertools.combinations(range(E), k)
                   if all(beats(row, a, b) for a in c for b in range(E) if b not in c)]
        assert len(winners) == 1
        assert set(ids[t]) == winners[0]
        for j in range(k - 1):
            assert beats(row, ids[t, j], ids[t, j + 1])


def test_topk_signed_zero_is_a_tie(oracle_mod):
    logits = np.array([[-0.0, 0.0, -1.0, -0.0], [0.0, -0.0, 0.0, 0.0]], dtype=np.float32)
    ids, w = oracle_mod.route_topk(logits, 3, renorm=True)
    assert ids.tolist() == [[0, 1, 3], [0, 1, 2]]
    np.testing.assert_allclose(w, np.full((2, 3), 1 / 3, dtype=np.float32), rtol=0, atol=0)


def test_topk_against_torch_on_tie_free_rows(oracle_mod):
    g = torch.Generator().manual_seed(3)
    logits = torch.randn((300, 128), generator=g)
    ids, w = oracle_mod.route_topk(logits.numpy(), 8, renorm=False)
    tv, ti = torch.topk(logits, 8, dim=1)  # tie-free: values are distinct
    assert np.array_equal(ids, ti.numpy().astype(np.int32))


# ---------------------------------------------------------------------------
# routing: weights
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("renorm", [False, True])
def test_weights_match_torch_softmax(oracle_mod, renorm):
    g = torch.Generator().manual_seed(5)
    logits = torch.randn((200, 64), generator=g) * 2
    k = 6
    ids, w = oracle_mod.route_topk(logits.numpy(), k, renorm)
    p = torch.softmax(logits.double(), dim=1).numpy()
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    if renorm:
        sel = sel / sel.sum(axis=1, keepdims=True)
    ref = sel.astype(np.float32)
    ulps = np.abs(w.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1


def test_weights_two_expert_closed_form(oracle_mod):
    # softmax over two logits is the logistic function of their difference
    a = np.linspace(-6, 6, 49, dtype=np.float32)
    b = np.float32(0.75)
    logits = np.stack([a, np.full_like(a, b)], axis=1)
    ids, w = oracle_mod.route_topk(logits, 2, renorm=False)
    for t in range(len(a)):
        pa = 1.0 / (1.0 + math.exp(float(b) - float(a[t])))
        want = {0: pa, 1: 1.0 - pa}
        for j in range(2):
            assert w[t, j] == np.float32(want[int(ids[t, j])])


def test_weights_uniform_and_sums(oracle_mod):
    E, k = 16, 4
    logits = np.full((3, E), 0.25, dtype=np.float32)
    ids, w = oracle_mod.route_topk(logits, k, renorm=False)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3
    assert np.all(w == np.float32(1 / E))
    ids, w = oracle_mod.route_topk(logits, k, renorm=True)
    assert np.all(w == np.float32(1 / k))
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((100, 32)).astype(np.float32)
    _, w_all = oracle_mod.route_topk(logits, 32, renorm=False)   # k = E: every probability
    np.testing.assert_allclose(w_all.astype(np.float64).sum(1), 1.0, atol=32 * 2 ** -24)
    _, w_rn = oracle_mod.route_topk(logits, 5, renorm=True)
    np.testing.assert_allclose(w_rn.astype(np.float64).sum(1), 1.0, atol=5 * 2 ** -24)


def test_weights_shift_invariance(oracle_mod):
    # softmax is invariant under adding a constant to every logit (exact here:
    # the shift is a power of two and the values stay exactly representable)
    rng = np.random.default_rng(2)
    logits = (rng.integers(-64, 64, size=(50, 16)) / 8).astype(np.float32)
    _, w0 = oracle_mod.route_topk(logits, 3, renorm=False)
    _, w1 = oracle_mod.route_topk(logits + np.float32(4.0), 3, renorm=False)
    assert np.array_equal(w0, w1)


# ---------------------------------------------------------------------------
# routing: permutation
# ---------------------------------------------------------------------------

def test_route_hand_worked_example(oracle_mod):
    fx = read_fixture("route_hand_worked.txt")
    T, E, k = int(fx["T"][0]), int(fx["E"][0]), int(fx["k"][0])
    logits = np.array([float(v) for v in fx["logits"]], dtype=np.float32).reshape(T, E)
    r = oracle_mod.route(logits, k, renorm=True)
    assert r["topk_ids"].ravel().tolist() == [int(v) for v in fx["topk_ids"]]
    assert r["expert_counts"].tolist() == [int(v) for v in fx["expert_counts"]]
    assert r["expert_offsets"].tolist() == [int(v) for v in fx["expert_offsets"]]
    assert r["perm"].tolist() == [int(v) for v in fx["perm"]]
    assert r["inv_perm"].tolist() == [int(v) for v in fx["inv_perm"]]
    # weights by closed form: t0 and t2 pick two equal logits -> 1/2 each;
    # t1 picks logits 3 and 1 -> logistic of their difference
    w = r["topk_weights"]
    assert w[0].tolist() == [0.5, 0.5] and w[2].tolist() == [0.5, 0.5]
    p = 1 / (1 + math.exp(-2.0))
    assert w[1].tolist() == [np.float32(p), np.float32(1 - p)]


def _check_perm_invariants(ids, E, counts, offsets, perm, inv_perm):
    S = ids.size
    flat = ids.ravel()
    assert np.array_equal(np.sort(perm), np.arange(S))              # bijection
    assert np.array_equal(inv_perm[perm], np.arange(S))             # inverse
    assert np.array_equal(perm[inv_perm], np.arange(S))
    assert np.array_equal(counts, np.bincount(flat, minlength=E))   # brute-force count
    assert counts.sum() == S
    assert offsets[0] == 0 and offsets[-1] == S
    assert np.array_equal(np.diff(offsets), counts)
    experts_along_p = flat[perm]
    assert np.all(np.diff(experts_along_p) >= 0)                    # expert-sorted
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                             # stable in slot order
    # the same permutation from a library stable sort
    assert np.array_equal(perm, np.argsort(flat, kind="stable").astype(np.int32))


@pytest.mark.parametrize("T,E,k,skew", [(1, 4, 2, 0), (7, 8, 2, 0), (257, 32, 4, 3.0),
                                         (64, 128, 8, 0), (100, 3, 3, 0), (50, 256, 1, 0)])
def test_permutation_invariants(oracle_mod, T, E, k, skew):
    rng = np.random.default_rng(T * 7 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, : min(4, E)] += skew
    r = oracle_mod.route(logits, k, renorm=True)
    _check_perm_invariants(r["topk_ids"], E, r["expert_counts"], r["expert_offsets"],
                           r["perm"], r["inv_perm"])


def test_permutation_all_tokens_one_expert(oracle_mod):
    T, E, k = 33, 16, 1
    logits = np.zeros((T, E), dtype=np.float32)
    logits[:, 9] = 5.0
    r = oracle_mod.route(logits, k, renorm=False)
    assert np.all(r["topk_ids"] == 9)
    assert r["expert_counts"][9] == T and r["expert_counts"].sum() == T
    assert np.array_equal(r["perm"], np.arange(T))


# ---------------------------------------------------------------------------
# expand
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,E,k", [(1, 8, 4, 2), (37, 64, 8, 2), (64, 256, 128, 8)])
def test_expand_round_trip(oracle_mod, T, H, E, k):
    rng = np.random.default_rng(T + H)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.integers(0, 2 ** 16, size=(T, H), dtype=np.uint16)   # any bit pattern, NaNs included
    r = oracle_mod.route(logits, k, renorm=True)
    ex = oracle_mod.expand(x, k, r["perm"])
    inv = r["inv_perm"].reshape(T, k)
    for j in range(k):
        assert np.array_equal(ex[inv[:, j]], x)                    # inverse permutation restores x
    assert np.array_equal(ex, x[r["perm"] // k])                   # numpy gather
    # a block of rows from an offset slice of perm
    p0, p1 = T // 3, T // 3 + 5
    assert np.array_equal(oracle_mod.expand(x, k, r["perm"][p0:p1]), ex[p0:p1])


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def _torch_swiglu_bits(oracle_mod, gate_up_bits):
    gu = bf16_bits_to_f64(gate_up_bits)
    I = gu.shape[1] // 2
    g = torch.from_numpy(gu[:, :I])
    u = torch.from_numpy(gu[:, I:])
    real = (torch.nn.functional.silu(g) * u).numpy()
    return oracle_mod.bf16_round(real)


def test_swiglu_matches_torch_silu(oracle_mod):
    g = torch.Generator().manual_seed(9)
    gu = (torch.randn((300, 2 * 96), generator=g) * 3).to(torch.bfloat16)
    bits = gu.view(torch.int16).numpy().view(np.uint16)
    ours = oracle_mod.swiglu(bits)
    ref = _torch_swiglu_bits(oracle_mod, bits)
    assert np.array_equal(ours, ref)


def test_swiglu_special_cases(oracle_mod):
    o = oracle_mod
    I = 64
    rng = np.random.default_rng(4)
    gate = (rng.standard_normal((4, I)) * 4).astype(np.float32)
    gate_b = o.bf16_round(gate.astype(np.float64))
    ones = np.full((4, I), 0x3F80, dtype=np.uint16)
    zeros = np.zeros((4, I), dtype=np.uint16)
    # up == 1: act is silu(gate) alone (gate is the FIRST half)
    act = o.swiglu(np.concatenate([gate_b, ones], axis=1))
    gd = bf16_bits_to_f64(gate_b)
    assert np.array_equal(act, o.bf16_round(gd / (1 + np.exp(-gd))))
    # swapping the halves must give something else: silu(1) * gate
    swapped = o.swiglu(np.concatenate([ones, gate_b], axis=1))
    assert not np.array_equal(swapped, act)
    assert np.array_equal(swapped, o.bf16_round(gd / (1 + math.exp(-1.0))))
    # up == 0 or gate == 0: zero
    assert np.all(bf16_bits_to_f64(o.swiglu(np.concatenate([gate_b, zeros], 1))) == 0)
    assert np.all(bf16_bits_to_f64(o.swiglu(np.concatenate([zeros, gate_b], 1))) == 0)
    # large positive gate: silu(g) = g exactly at bfloat16 precision
    big = o.bf16_round(np.full((1, I), 60.0))
    assert np.array_equal(o.swiglu(np.concatenate([big, ones[:1]], 1)), big)
    # large negative gate: silu(g) is far below the smallest bfloat16 -> -0
    neg = o.bf16_round(np.full((1, I), -120.0))
    assert np.all(o.swiglu(np.concatenate([neg, ones[:1]], 1)) == 0x8000)
    # silu(-1) * 2 = -2 / (1 + e), a closed form
    v = o.swiglu(np.concatenate([o.bf16_round(np.full((1, I), -1.0)),
                                 o.bf16_round(np.full((1, I), 2.0))], 1))
    assert np.all(v == o.bf16_round(np.array([-2.0 / (1.0 + math.e)]))[0])


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

def _routed_case(oracle_mod, T, H, E, k, renorm=True, seed=0):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = oracle_mod.bf16_round(rng.standard_normal((T, H)))
    r = oracle_mod.route(logits, k, renorm)
    return x, r


@pytest.mark.parametrize("T,H,E,k", [(5, 16, 4, 2), (64, 256, 8, 2), (40, 128, 128, 8), (9, 64, 32, 16)])
def test_combine_identity_expert_returns_x(oracle_mod, T, H, E, k):
    # expert_out = expanded_x with renormalised weights: sum_j w_j x = x*(1 +- k 2^-24),
    # which rounds back to x exactly
    x, r = _routed_case(oracle_mod, T, H, E, k)
    ex = oracle_mod.expand(x, k, r["perm"])
    out = oracle_mod.combine(ex, r["topk_weights"], r["inv_perm"])
    assert np.array_equal(out, x)


def test_combine_single_expert_unit_weight_is_a_gather(oracle_mod):
    T, H, E, k = 30, 32, 8, 1
    x, r = _routed_case(oracle_mod, T, H, E, k)
    rng = np.random.default_rng(1)
    eo = oracle_mod.bf16_round(rng.standard_normal((T, H)))
    out = oracle_mod.combine(eo, np.ones((T, 1), np.float32), r["inv_perm"])
    assert np.array_equal(out, eo[r["inv_perm"]])


def test_combine_zero_weights_and_scaling(oracle_mod):
    T, H, E, k = 20, 48, 16, 4
    x, r = _routed_case(oracle_mod, T, H, E, k, seed=3)
    rng = np.random.default_rng(5)
    eo = oracle_mod.bf16_round(rng.standard_normal((T * k, H)))
    z = oracle_mod.combine(eo, np.zeros((T, k), np.float32), r["inv_perm"])
    assert np.all(bf16_bits_to_f64(z) == 0)
    w = r["topk_weights"]
    o1 = bf16_bits_to_f64(oracle_mod.combine(eo, w, r["inv_perm"]))
    o2 = bf16_bits_to_f64(oracle_mod.combine(eo, 2 * w, r["inv_perm"]))
    assert np.array_equal(o2, 2 * o1)   # power-of-two scaling commutes with rounding


def test_combine_matches_numpy_weighted_sum(oracle_mod):
    T, H, E, k = 64, 96, 32, 4
    x, r = _routed_case(oracle_mod, T, H, E, k, seed=8)
    rng = np.random.default_rng(6)
    eo = oracle_mod.bf16_round(rng.standard_normal((T * k, H)) * 2)
    w = r["topk_weights"]
    rows = bf16_bits_to_f64(eo)[r["inv_perm"].reshape(T, k)]        # [T, k, H] gather
    real = np.einsum("tk,tkh->th", w.astype(np.float64), rows)
    ref = oracle_mod.bf16_round(real)
    ours = oracle_mod.combine(eo, w, r["inv_perm"])
    assert bf16_ulp_distance(ours, ref).max() <= 1
    assert (ours == ref).mean() > 0.999
    # a token sub-range through offset slices
    t0, t1 = 10, 20
    part = oracle_mod.combine(eo, w[t0:t1], r["inv_perm"][t0 * k:t1 * k])
    assert np.array_equal(part, ours[t0:t1])


# ---------------------------------------------------------------------------
# local (expert-range) routing with padded segments
# ---------------------------------------------------------------------------

def test_route_local_hand_worked_example(oracle_mod):
    base = read_fixture("route_hand_worked.txt")
    fx = read_fixture("route_local_hand_worked.txt")
    T, E, k = int(base["T"][0]), int(base["E"][0]), int(base["k"][0])
    ids = np.array([int(v) for v in base["topk_ids"]], dtype=np.int32).reshape(T, k)
    e0, e1, pad, rows = (int(fx[n][0]) for n in ("e0", "e1", "pad", "rows"))
    counts, offsets, perm, inv = oracle_mod.route_permute_local(ids, E, e0, e1, pad, rows)
    assert counts.tolist() == [int(v) for v in fx["counts"]]
    assert offsets.tolist() == [int(v) for v in fx["offsets"]]
    assert perm.tolist() == [int(v) for v in fx["perm"]]
    assert inv.tolist() == [int(v) for v in fx["inv_perm"]]
    assert oracle_mod.local_rows_capacity(T, k, e1 - e0, pad) == rows


@pytest.mark.parametrize("T,E,k", [(37, 8, 2), (200, 64, 8), (129, 32, 4)])
def test_route_local_full_range_without_padding_is_the_full_routing(oracle_mod, T, E, k):
    rng = np.random.default_rng(T)
    r = oracle_mod.route(rng.standard_normal((T, E)).astype(np.float32), k, True)
    counts, offsets, perm, inv = oracle_mod.route_permute_local(r["topk_ids"], E, 0, E, 1)
    assert np.array_equal(counts, r["expert_counts"])
    assert np.array_equal(offsets, r["expert_offsets"])
    assert np.array_equal(perm, r["perm"])
    assert np.array_equal(inv, r["inv_perm"])


@pytest.mark.parametrize("pad", [1, 4, 128])
def test_route_local_partition_matches_global_segments(oracle_mod, pad):
    # split the experts into ranges (ranks); every rank's rows in order are the
    # global permutation's segment for its experts, padding aside
    T, E, k = 300, 32, 4
    rng = np.random.default_rng(pad)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, :3] += 2.0
    r = oracle_mod.route(logits, k, True)
    g_off = r["expert_offsets"]
    seen = np.zeros(T * k, dtype=int)
    for e0, e1 in [(0, 5), (5, 6), (6, 20), (20, 32)]:
        counts, offsets, perm, inv = oracle_mod.route_permute_local(r["topk_ids"], E, e0, e1, pad)
        assert np.array_equal(counts, r["expert_counts"][e0:e1])
        assert np.all(offsets % pad == 0)
        slack = np.diff(offsets) - counts
        assert np.all((slack >= 0) & (slack < pad))
        rows_used = perm[perm >= 0]
        assert np.array_equal(rows_used, r["perm"][g_off[e0]:g_off[e1]])
        local = (r["topk_ids"].ravel() >= e0) & (r["topk_ids"].ravel() < e1)
        assert np.all(inv[~local] == -1)
        assert np.array_equal(perm[inv[local]], np.flatnonzero(local))
        for l in range(e1 - e0):                          # padding rows are -1
            assert np.all(perm[offsets[l] + counts[l]:offsets[l + 1]] == -1)
        assert np.all(perm[offsets[-1]:] == -1)
        seen[local] += 1
    assert np.all(seen == 1)                              # every slot on exactly one rank


def test_combine_partial_sums_skip_other_ranks(oracle_mod):
    # a rank's partial combine (-1 for slots it does not hold) equals the full
    # combine with the other ranks' weights set to zero, and the partials of
    # all ranks add up (in real arithmetic) to the full combine
    T, H, E, k = 40, 64, 16, 4
    rng = np.random.default_rng(3)
    r = oracle_mod.route(rng.standard_normal((T, E)).astype(np.float32), k, True)
    eo_full = oracle_mod.bf16_round(rng.standard_normal((T * k, H)))
    ids = r["topk_ids"]
    total = np.zeros((T, H))
    mag = np.zeros((T, H))
    for e0, e1 in [(0, 7), (7, 16)]:
        counts, offsets, perm, inv = oracle_mod.route_permute_local(ids, E, e0, e1, 8)
        eo = np.zeros((perm.size, H), dtype=np.uint16)
        eo[perm >= 0] = eo_full[r["inv_perm"][perm[perm >= 0]]]   # each local row's data
        part = oracle_mod.combine(eo, r["topk_weights"], inv)
        w0 = r["topk_weights"] * ((ids >= e0) & (ids < e1))
        assert np.array_equal(part, oracle_mod.combine(eo_full, w0, r["inv_perm"]))
        total += bf16_bits_to_f64(part)
        mag += np.abs(bf16_bits_to_f64(part))
    full = bf16_bits_to_f64(oracle_mod.combine(eo_full, r["topk_weights"], r["inv_perm"]))
    # each partial and the full result are rounded once (half a bf16 ulp each)
    assert np.all(np.abs(total - full) <= 2 ** -8 * (mag + np.abs(full)))


# ---------------------------------------------------------------------------
# MXFP8 (E4M3 elements, E8M0 scale per 32)
# ---------------------------------------------------------------------------

def test_e4m3_round_known_patterns(oracle_mod):
    cases = [(448.0, 0x7E), (1.0, 0x38), (0.5, 0x30), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01),
             (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (464.0, 0x7E), (1e9, 0x7E), (-448.0, 0xFE),
             (1.0625, 0x38), (1.1875, 0x3A), (0.0, 0x00), (-0.0, 0x80), (240.0, 0x77),
             (7 * 2.0 ** -9, 0x07), (-3.0, 0xC4), (math.inf, 0x7E)]   # -3 = -1.5*2^1: 0x80|8<<3|4
    got = oracle_mod.e4m3_round(np.array([v for v, _ in cases]))
    assert [int(g) for g in got] == [b for _, b in cases]


def test_e4m3_matches_torch_in_range(oracle_mod):
    fp8 = getattr(torch, "float8_e4m3fn", None)
    if fp8 is None:
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100_000) * 50, rng.standard_normal(20_000) * 1e-2,
                        rng.uniform(-448, 448, 20_000)]).astype(np.float32)
    ours = oracle_mod.e4m3_round(v.astype(np.float64))
    ref = torch.from_numpy(v).to(fp8).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle_mod.e4m3_decode(codes)
    tref = torch.from_numpy(codes).view(fp8).to(torch.float64).numpy()
    nan = np.isnan(tref)
    assert np.array_equal(np.isnan(dec), nan)
    np.testing.assert_array_equal(dec[~nan], tref[~nan])


def test_mxfp8_scales_closed_forms(oracle_mod):
    O = oracle_mod
    rows = np.zeros((5, 64))
    rows[0, :32] = 448.0                   # amax 448: X = 0, byte 127, codes 0x7E
    rows[0, 32:] = 0.0                     # zero block: byte 0, codes 0
    rows[1, :32] = 1.0                     # amax 1: X = -8, 1 / 2^-8 = 256 = 0x78
    rows[1, 32:] = np.linspace(-0.75, 0.75, 32)   # amax 0.75: X = -9
    rows[2, :32] = 2.0 ** -130             # tiny (bf16 subnormal): X clamps to -127
    rows[2, 32:] = 500.0                   # amax 500: X = 0; 500 saturates to 448
    rows[3, :] = np.arange(64) - 31.5      # amax 31.5 / 32: X = -4
    rows[4, :] = 3.0e38                    # near the top of the bf16 range: X = 119
    x = O.bf16_round(rows)
    codes, scales = O.quant_mxfp8(x)
    assert scales.tolist() == [[127, 0], [119, 118], [0, 127], [123, 123], [246, 246]]
    assert np.all(codes[0, :32] == 0x7E) and np.all(codes[0, 32:] == 0)
    assert np.all(codes[1, :32] == 0x78)
    assert np.all(codes[2, 32:] == 0x7E)
    assert np.all(codes[2, :32] == O.e4m3_round(np.full(32, 2.0 ** -130 * 2.0 ** 127)))


def test_mxfp8_round_trip_error_bound(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(1)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-12, 12, (64, 1)))
    x = O.bf16_round(v)
    xv = O.bf16_decode(x)
    codes, scales = O.quant_mxfp8(x)
    deq = O.dequant_mxfp8(codes, scales)
    X = np.repeat(scales.astype(np.float64) - 127, 32, axis=1)
    scaled = np.abs(xv) / 2.0 ** X
    # every block's largest magnitude lands in [256, 512)
    amax_scaled = scaled.reshape(64, 8, 32).max(axis=2)
    assert np.all((amax_scaled >= 256) & (amax_scaled < 512))
    inside = scaled <= 448
    # half an E4M3 ulp: 2^-4 relative for normals, 2^-10 * 2^X for subnormals
    bound = np.maximum(2.0 ** -4 * np.abs(xv), 2.0 ** (X - 10))
    assert np.all(np.abs(deq - xv)[inside] <= bound[inside])
    assert np.all(np.abs(deq[~inside]) == 448 * 2.0 ** X[~inside])
    assert np.all(np.sign(deq) * np.sign(xv) >= 0)


# ---------------------------------------------------------------------------
# FP4 (E2M1) block quantization: MXFP4 and NVFP4
# ---------------------------------------------------------------------------

# The E2M1 value of every code, as tabulated by the OCP Microscaling v1.0
# specification (sign bit 0x8; exponent bias 1; 0.5 is the one subnormal).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decode_table(oracle_mod):
    got = oracle_mod.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert got.tolist() == E2M1_TABLE
    assert np.all(np.signbit(got[8:]))


def test_e2m1_round_known_patterns(oracle_mod):
    cases = [  # value, code: exact values, ties to the even code, saturation, sign
        (0.0, 0x0), (0.5, 0x1), (1.0, 0x2), (1.5, 0x3), (2.0, 0x4), (3.0, 0x5), (4.0, 0x6), (6.0, 0x7),
        (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
        (0.2499, 0x0), (0.2501, 0x1), (0.7499, 0x1), (0.7501, 0x2), (2.4999, 0x4), (2.5001, 0x5),
        (4.9999, 0x6), (5.0001, 0x7), (7.0, 0x7), (100.0, 0x7), (1e-30, 0x0),
        (-0.1, 0x8), (-0.0, 0x8), (-0.3, 0x9), (-1.0, 0xA), (-5.0, 0xE), (-6.0, 0xF), (-1e9, 0xF),
    ]
    got = oracle_mod.e2m1_round(np.array([v for v, _ in cases]))
    assert got.tolist() == [c for _, c in cases]


def test_e2m1_round_is_nearest_with_even_ties(oracle_mod):
    """Brute force: the nearest of the 8 magnitudes (the even code on a tie),
    for a sweep that hits every midpoint."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.uniform(-7.5, 7.5, 20000), np.arange(-6.5, 6.5001, 0.125)])
    got = oracle_mod.e2m1_round(v)
    for x, c in zip(v, got):
        d = np.abs(np.abs(x) - mags)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        if abs(x) >= 6:
            want = 7
        assert c == (want | (0x8 if np.signbit(x) else 0)), (x, c, want)


def test_fp4_nibble_packing(oracle_mod):
    O = oracle_mod
    x = O.bf16_round(np.array([[1.0, 6.0, -0.5, 2.0] + [0.0] * 28]))   # amax 6: X = 0
    codes, scales = O.quant_mxfp4(x)
    assert scales.tolist() == [[127]]
    assert codes[0, :2].tolist() == [0x72, 0x49]    # element 2i in the low nibble


def test_mxfp4_scales_closed_forms(oracle_mod):
    O = oracle_mod
    rows = np.zeros((5, 64))
    rows[0, :32] = 6.0                        # amax 6: X = floor(log2 6) - 2 = 0, codes 0x7
    rows[0, 32:] = 0.0                        # zero block: X = -127, byte 0, codes 0
    rows[1, :32] = 1.0                        # amax 1: X = -2, 1 * 4 = 4 -> 0x6
    rows[1, 32:] = np.linspace(-0.75, 0.75, 32)   # amax 0.75: X = -3
    rows[2, :32] = 2.0 ** -130                # X clamps to -127: 2^-3 rounds to 0
    rows[2, 32:] = 7.0                        # amax 7: X = 0; 7 saturates to 6
    rows[3, :] = np.arange(64) - 31.5         # amax 31.5 / 32: X = 2
    rows[4, :] = 3.0e38                       # top of the bf16 range: X = 127 - 2
    x = O.bf16_round(rows)
    codes, scales = O.quant_mxfp4(x)
    assert scales.tolist() == [[127, 0], [125, 124], [0, 127], [129, 129], [252, 252]]
    c = O.unpack_fp4(codes)
    assert np.all(c[0, :32] == 0x7) and np.all(c[0, 32:] == 0)
    assert np.all(c[1, :32] == 0x6)
    assert np.all(c[2, :32] == 0x0) and np.all(c[2, 32:] == 0x7)
    # 0.75 * 2^3 = 6 -> 0x7 at the ends of the linspace block
    assert c[1, 32] == 0xF and c[1, 63] == 0x7


def test_mxfp4_round_trip_error_bound(oracle_mod):
    O = oracle_mod
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-12, 12, (64, 1)))
    x = O.bf16_round(v)
    xv = O.bf16_decode(x)
    codes, scales = O.quant_mxfp4(x)
    deq = O.dequant_mxfp4(codes, scales)
    X = np.repeat(scales.astype(np.float64) - 127, 32, axis=1)
    scaled = np.abs(xv) / 2.0 ** X
    amax_scaled = scaled.reshape(64, 8, 32).max(axis=2)
    assert np.all((amax_scaled >= 4) & (amax_scaled < 8))   # amax lands in [4, 8)
    inside = scaled <= 6
    # half the E2M1 spacing: at most 1 (between 4 and 6), in units of 2^X
    assert np.all(np.abs(deq - xv)[inside] <= 2.0 ** X[inside])
    assert np.all(np.abs(deq[~inside]) == 6 * 2.0 ** X[~inside])
    assert np.all(np.sign(deq) * np.sign(xv) >= 0)


def test_nvfp4_closed_forms(oracle_mod):
    O = oracle_mod
    rows = np.zeros((3, 32))
    rows[0, :16] = [6.0, -3.0, 1.0, 0.5] + [0.0] * 12   # g = 1: scale E4M3(1) = 0x38, codes = E2M1(v)
    rows[0, 16:] = 0.0                                  # zero block: scale 0, codes 0
    rows[1, :16] = 12.0                                 # g = 1: t = 12/6 = 2 -> 0x40; v * 1/2 = 6
    rows[1, 16:] = np.linspace(-3.0, 3.0, 16)           # amax 3: scale E4M3(0.5) = 0x30
    rows[2, :] = 1000.0                                 # g = 1: 1000/6 = 166.67 -> E4M3 160 = 1.25 * 2^7 (0x72)
    x = O.bf16_round(rows)
    codes, scales = O.quant_nvfp4(x, 1.0)
    assert scales.tolist() == [[0x38, 0x00], [0x40, 0x30], [0x72, 0x72]]
    c = O.unpack_fp4(codes)
    assert c[0, :4].tolist() == [0x7, 0xD, 0x2, 0x1] and np.all(c[0, 4:] == 0)
    assert np.all(c[1, :16] == 0x7)
    assert c[1, 16] == 0xF and c[1, 31] == 0x7            # +-3 / 0.5 = +-6
    # 1000 * (1 / 160) = 6.25 saturates to 6
    assert np.all(c[2] == 0x7)
    # a calibrated tensor scale g = 448 * 6 / amax puts the largest block's
    # scale at E4M3's top (448) and its largest value at code 6
    xv = O.bf16_decode(x[1:2])
    g = 448.0 * 6.0 / np.abs(xv).max()
    codes, scales = O.quant_nvfp4(x[1:2], g)
    assert scales[0, 0] == 0x7E and np.all(O.unpack_fp4(codes)[0, :16] == 0x7)


@pytest.mark.parametrize("g", [1.0, 0.37, 448.0 * 6.0 / 9.0])
def test_nvfp4_round_trip_error_bound(oracle_mod, g):
    O = oracle_mod
    rng = np.random.default_rng(3)
    v = rng.standard_normal((32, 128)) * np.exp(rng.uniform(-3, 3, (32, 1)))
    x = O.bf16_round(v)
    xv = O.bf16_decode(x)
    codes, scales = O.quant_nvfp4(x, g)
    deq = O.dequant_nvfp4(codes, scales, g)
    s = np.repeat(O.e4m3_decode(scales), 16, axis=1)
    unit = s / g                      # the value of E2M1 1.0 in this block
    scaled = np.abs(xv) / unit
    inside = scaled <= 6
    # within half the largest E2M1 spacing (1 unit); beyond 6 units, saturated
    assert np.all(np.abs(deq - xv)[inside] <= unit[inside] * (1 + 1e-6))
    assert np.all(np.abs(deq[~inside]) == 6 * unit[~inside])
    # where g * amax / 6 lies in E4M3's normal range (2^-6 .. 448), its
    # rounding is within 2^-4 relative, so the block's largest value lands
    # at most 6 / (1 - 2^-4) after scaling
    raw = g * np.abs(xv).reshape(32, 8, 16).max(axis=2) / 6
    normal = np.repeat((raw >= 2.0 ** -6) & (raw <= 448), 16, axis=1)
    assert np.all(scaled[normal] <= 6 / (1 - 2.0 ** -4) * (1 + 1e-6))
    assert np.all(np.sign(deq) * np.sign(xv) >= 0)


# ---------------------------------------------------------------------------
# QK RMSNorm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("hd", [64, 128, 256])
def test_rmsnorm_matches_torch_rms_norm(oracle_mod, hd):
    O = oracle_mod
    rng = np.random.default_rng(hd)
    x = O.bf16_round(rng.standard_normal((200, hd)) * np.exp(rng.uniform(-3, 3, (200, 1))))
    w = O.bf16_round(rng.standard_normal(hd) * 0.1)
    bias, eps = 1.0, 1e-6
    xt = torch.from_numpy(O.bf16_decode(x))
    wt = torch.from_numpy(O.bf16_decode(w)) + bias
    ref = torch.nn.functional.rms_norm(xt, (hd,), wt, eps).numpy()
    assert np.array_equal(O.rmsnorm_heads(x, w, bias, eps), O.bf16_round(ref))


def test_rmsnorm_closed_forms(oracle_mod):
    O = oracle_mod
    hd = 128
    one = O.bf16_round(np.ones(hd))
    zero_w = O.bf16_round(np.zeros(hd))
    # a constant head c with eps = 0: x / rms(x) = sign(c); with w = 0, bias 1
    for c in (3.0, -0.25, 1e-20):
        x = O.bf16_round(np.full((1, hd), c))
        assert np.all(O.bf16_decode(O.rmsnorm_heads(x, zero_w, 1.0, 0.0)) == np.sign(c))
    # the weight multiplies, the bias adds to it: w = 1, bias = 0.5 -> 1.5 * sign
    x = O.bf16_round(np.full((1, hd), -7.0))
    assert np.all(O.bf16_decode(O.rmsnorm_heads(x, one, 0.5, 0.0)) == -1.5)
    # a head of +-1 alternating with eps = 3: 1 / sqrt(1 + 3) = 0.5
    x = O.bf16_round(np.tile([1.0, -1.0], hd // 2)[None, :])
    assert np.all(O.bf16_decode(O.rmsnorm_heads(x, zero_w, 1.0, 3.0)) == np.tile([0.5, -0.5], hd // 2))
    # scale invariance (eps = 0, power-of-two scale: exact)
    rng = np.random.default_rng(4)
    x = O.bf16_round(rng.standard_normal((50, hd)))
    x8 = O.bf16_round(O.bf16_decode(x) * 8.0)
    w = O.bf16_round(rng.standard_normal(hd))
    assert np.array_equal(O.rmsnorm_heads(x, w, 0.0, 0.0), O.rmsnorm_heads(x8, w, 0.0, 0.0))
    # every head is normalised on its own: one head's values do not leak
    xx = x.copy()
    xx[7] = O.bf16_round(rng.standard_normal(hd) * 1000)
    a, b = O.rmsnorm_heads(x, w, 0.0, 1e-6), O.rmsnorm_heads(xx, w, 0.0, 1e-6)
    assert np.array_equal(np.delete(a, 7, 0), np.delete(b, 7, 0))
