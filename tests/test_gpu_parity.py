"""CUDA path against the CPU oracle, element by element, through the C ABI.

Bar: top-k ids, counts, offsets, perm, inv_perm and expanded rows bit-exact;
SwiGLU and combine outputs within |gpu - ref| <= 2e-2 + 1e-2 |ref|; routing
weights within 1e-7 + 1e-5 |ref| (see helpers.py for the derivations).
Inputs are seeded and synthetic; both sides get the same host bytes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import (check_bf16_close, check_exact, check_weights_close)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_moe_gb300 import build
    build.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def O(oracle_mod):
    return oracle_mod


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


_CACHE = {}


def workload_inputs(name):
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    if name not in _CACHE:
        w = WORKLOADS[name]
        _CACHE[name] = (w, generate(w, seed=0))
    return _CACHE[name]


def gpu_route(dev, logits_np, k, renorm):
    from memory_bound_moe_gb300 import moe_route
    r = moe_route(torch.from_numpy(np.ascontiguousarray(logits_np)).to(dev), k, renorm)
    torch.cuda.synchronize()
    return {f: getattr(r, f).cpu().numpy() for f in r._fields}


def assert_route_equal(got, ref, what):
    check_exact(got["topk_ids"], ref["topk_ids"], f"{what} topk_ids")
    check_exact(got["expert_counts"], ref["expert_counts"], f"{what} counts")
    check_exact(got["expert_offsets"], ref["expert_offsets"], f"{what} offsets")
    check_exact(got["perm"], ref["perm"], f"{what} perm")
    check_exact(got["inv_perm"], ref["inv_perm"], f"{what} inv_perm")
    check_weights_close(got["topk_weights"], ref["topk_weights"], f"{what} weights")


CONFIGS = ["tiny", "mid", "decode", "prefill", "skewed"]


# ---------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", CONFIGS)
def test_route_workload(dev, O, name):
    w, inp = workload_inputs(name)
    logits = inp["logits"].numpy()
    ref = O.route(logits, w.k, w.renorm)
    got = gpu_route(dev, logits, w.k, w.renorm)
    assert_route_equal(got, ref, name)


@pytest.mark.parametrize("name", CONFIGS)
def test_expand_workload(dev, O, name):
    from memory_bound_moe_gb300 import moe_expand
    w, inp = workload_inputs(name)
    ref_r = O.route(inp["logits"].numpy(), w.k, w.renorm)
    x = u16(inp["x"])
    out = torch.full((w.S, w.H), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)  # canary 0xFFFF
    moe_expand(bf16_dev(x, dev), torch.from_numpy(ref_r["inv_perm"]).to(dev), w.k, out=out)
    torch.cuda.synchronize()
    check_exact(u16(out), O.expand(x, w.k, ref_r["perm"]), f"{name} expanded_x")


@pytest.mark.parametrize("name", CONFIGS)
def test_swiglu_workload(dev, oracle_act, name):
    """Every element of every workload's act, prefill's 16384 x 14336
    included (compared in chunks)."""
    from memory_bound_moe_gb300 import moe_swiglu
    gu, ref = oracle_act(name)
    act = u16(moe_swiglu(bf16_dev(gu, dev)))
    stats = check_bf16_close(act, ref, f"{name} act")
    # one float32 evaluation rounded once: nearly every element is the
    # correctly rounded value
    assert stats["exact_frac"] > 0.999, stats


@pytest.mark.parametrize("name", CONFIGS)
def test_combine_workload(dev, O, name):
    from memory_bound_moe_gb300 import moe_combine
    w, inp = workload_inputs(name)
    ref_r = O.route(inp["logits"].numpy(), w.k, w.renorm)
    eo = u16(inp["expert_out"])
    out = moe_combine(bf16_dev(eo, dev), torch.from_numpy(ref_r["topk_weights"]).to(dev),
                      torch.from_numpy(ref_r["inv_perm"]).to(dev))
    stats = check_bf16_close(u16(out), O.combine(eo, ref_r["topk_weights"], ref_r["inv_perm"]),
                             f"{name} out")
    # float32 accumulation then one rounding: nearly every element is the
    # correctly rounded value (bf16-ulp counts are meaningless where the k
    # terms cancel to a tiny sum, so the bound above is the criterion)
    assert stats["exact_frac"] > 0.98, stats


@pytest.mark.parametrize("name", CONFIGS)
def test_whole_path_workload(dev, O, oracle_act, name):
    """route -> expand -> SwiGLU -> combine on the GPU, each stage fed by the
    GPU's previous stage, against the oracle's path on the same inputs; every
    output compared in full."""
    from memory_bound_moe_gb300 import moe_combine, moe_expand, moe_route, moe_swiglu
    w, inp = workload_inputs(name)
    logits = inp["logits"].to(dev)
    x = inp["x"].to(dev)
    r = moe_route(logits, w.k, w.renorm)
    ex = moe_expand(x, r.inv_perm, w.k)
    act = moe_swiglu(inp["gate_up"].to(dev))
    out = moe_combine(inp["expert_out"].to(dev), r.topk_weights, r.inv_perm)
    torch.cuda.synchronize()
    ref = O.route(inp["logits"].numpy(), w.k, w.renorm)
    assert_route_equal({f: getattr(r, f).cpu().numpy() for f in r._fields}, ref, name)
    check_exact(u16(ex), O.expand(u16(inp["x"]), w.k, ref["perm"]), f"{name} expanded_x")
    del ex
    gu, ref_act = oracle_act(name)
    assert np.array_equal(gu, u16(inp["gate_up"]))
    check_bf16_close(u16(act), ref_act, f"{name} act")
    del act
    check_bf16_close(u16(out), O.combine(u16(inp["expert_out"]), ref["topk_weights"],
                                         ref["inv_perm"]), f"{name} out")


# ---------------------------------------------------------------------------
# routing edge cases (one-block and two-kernel paths)
# ---------------------------------------------------------------------------

ROUTE_CASES = [
    # T, E, k, renorm, kind
    (1, 8, 2, True, "normal"), (1, 1024, 16, False, "normal"), (7, 3, 3, True, "normal"),
    (31, 32, 4, True, "ties"), (33, 32, 4, False, "ties"), (64, 64, 1, True, "normal"),
    (65, 64, 8, True, "ties"), (256, 8, 2, True, "normal"), (257, 8, 8, False, "ties"),
    (257, 16, 5, True, "normal"), (1000, 17, 3, True, "normal"), (1023, 100, 6, True, "ties"),
    (2048, 256, 8, False, "normal"), (5000, 5, 2, True, "ties"), (3000, 512, 16, True, "normal"),
    (4099, 1024, 16, True, "normal"), (20000, 128, 8, True, "normal"), (70000, 8, 2, True, "normal"),
    (129, 2, 2, True, "ties"), (300, 1, 1, True, "normal"),
    # two tokens per warp step in the rank kernel: 256 and 160 experts (8 keys
    # per lane), and odd token runs per warp (3 and 47 tokens) with rounds
    # past the register-held ones
    (8192, 256, 8, True, "normal"), (40001, 160, 6, False, "ties"), (6000, 100, 4, True, "normal"),
    (94000, 64, 2, True, "ties"),
    # 1024-thread rank blocks (one token per warp): a ragged last block, and
    # 8 keys per lane with ties
    (3000, 100, 6, True, "normal"), (4096, 256, 8, False, "ties"),
]


def _logits(T, E, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "ties":
        l = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
        l[rng.random((T, E)) < 0.15] = -0.0
        return l
    return rng.standard_normal((T, E)).astype(np.float32)


@pytest.mark.parametrize("T,E,k,renorm,kind", ROUTE_CASES)
def test_route_edge_cases(dev, O, T, E, k, renorm, kind):
    logits = _logits(T, E, kind, seed=T * 31 + E)
    assert_route_equal(gpu_route(dev, logits, k, renorm), O.route(logits, k, renorm),
                       f"T={T} E={E} k={k}")


def test_route_all_tokens_one_expert_and_extremes(dev, O):
    T, E, k = 3000, 64, 4
    logits = np.zeros((T, E), dtype=np.float32)
    logits[:, 17] = 30.0
    logits[:, 3] = 20.0
    logits[::7, 40] = -1e30
    logits[::5, 41] = 1e30
    for renorm in (False, True):
        assert_route_equal(gpu_route(dev, logits, k, renorm), O.route(logits, k, renorm), "extreme")


def test_route_is_deterministic(dev):
    logits = _logits(5000, 128, "ties", seed=1)
    a = gpu_route(dev, logits, 8, True)
    b = gpu_route(dev, logits, 8, True)
    for f in a:
        assert np.array_equal(a[f], b[f]), f


def test_route_empty_batch(dev):
    from memory_bound_moe_gb300 import moe_route
    r = moe_route(torch.empty((0, 16), dtype=torch.float32, device=dev), 2, True)
    torch.cuda.synchronize()
    assert r.expert_counts.cpu().tolist() == [0] * 16
    assert r.expert_offsets.cpu().tolist() == [0] * 17


def test_route_reused_workspace_and_stream(dev, O):
    from memory_bound_moe_gb300 import moe_route, moe_route_workspace_size
    T, E, k = 4096, 128, 8
    ws = torch.full((moe_route_workspace_size(T, E, k),), 0x5A, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    for seed in range(3):
        logits = _logits(T, E, "normal", seed)
        with torch.cuda.stream(s):
            r = moe_route(torch.from_numpy(logits).to(dev), k, True, workspace=ws, stream=s)
        s.synchronize()
        assert_route_equal({f: getattr(r, f).cpu().numpy() for f in r._fields},
                           O.route(logits, k, True), f"seed {seed}")


# ---------------------------------------------------------------------------
# row kernels: odd shapes, both vector widths, special values
# ---------------------------------------------------------------------------

def _rand_bf16(O, shape, seed, scale=1.0):
    return O.bf16_round(np.random.default_rng(seed).standard_normal(shape) * scale)


def _offset16(t: torch.Tensor) -> torch.Tensor:
    """The same values at an address that is 16- but not 32-byte aligned
    (forces the 128-bit path)."""
    flat = torch.empty(t.numel() + 16, dtype=t.dtype, device=t.device)
    base = flat.data_ptr() % 32
    shift = ((16 - base) % 32) // t.element_size()
    view = flat[shift:shift + t.numel()].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 32 == 16
    return view


@pytest.mark.parametrize("rows,I", [(1, 8), (3, 16), (5, 24), (1000, 120), (77, 2880), (4096, 768),
                                    (2, 16384)])
@pytest.mark.parametrize("wide", [True, False])
def test_swiglu_shapes(dev, O, rows, I, wide):
    from memory_bound_moe_gb300 import moe_swiglu
    gu = _rand_bf16(O, (rows, 2 * I), seed=rows + I, scale=3.0)
    g = bf16_dev(gu, dev)
    if not wide:
        g = _offset16(g)
    check_bf16_close(u16(moe_swiglu(g)), O.swiglu(gu), f"rows={rows} I={I}")


def test_swiglu_special_values(dev, O):
    from memory_bound_moe_gb300 import moe_swiglu
    I = 64
    vals = np.array([0.0, -0.0, 1.0, -1.0, 10.0, -10.0, 40.0, -40.0, 87.0, -87.0, 88.5, -88.5,
                     100.0, -100.0, 3e38, -3e38, 1e-30, -1e-30, 0.5, -0.5], dtype=np.float64)
    gate = np.resize(vals, (len(vals), I))
    up = np.resize(vals[::-1], (len(vals), I))
    gu = np.concatenate([O.bf16_round(gate), O.bf16_round(up)], axis=1)
    ref = O.swiglu(gu)
    got = u16(moe_swiglu(bf16_dev(gu, dev)))
    fin = np.isfinite(O.bf16_decode(ref))
    check_bf16_close(got[fin], ref[fin], "special values")


@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (3, 16, 2), (17, 24, 3), (100, 264, 5), (33, 2880, 4),
                                   (9, 7168, 8), (5, 512, 16), (2000, 1024, 2)])
@pytest.mark.parametrize("wide", [True, False])
def test_expand_combine_shapes(dev, O, T, H, k, wide):
    from memory_bound_moe_gb300 import moe_combine, moe_expand
    E = max(k, 8)
    logits = _logits(T, E, "normal", seed=T + H)
    r = O.route(logits, k, True)
    x = _rand_bf16(O, (T, H), seed=H)
    eo = _rand_bf16(O, (T * k, H), seed=H + 1, scale=2.0)
    xd, eod = bf16_dev(x, dev), bf16_dev(eo, dev)
    if not wide:
        xd, eod = _offset16(xd), _offset16(eod)
    inv = torch.from_numpy(r["inv_perm"]).to(dev)
    ex = moe_expand(xd, inv, k, out=(None if wide else _offset16(torch.zeros((T * k, H), dtype=torch.bfloat16, device=dev))))
    out = moe_combine(eod, torch.from_numpy(r["topk_weights"]).to(dev), inv,
                      out=(None if wide else _offset16(torch.zeros((T, H), dtype=torch.bfloat16, device=dev))))
    check_exact(u16(ex), O.expand(x, k, r["perm"]), f"expand T={T} H={H} k={k}")
    check_bf16_close(u16(out), O.combine(eo, r["topk_weights"], r["inv_perm"]), f"combine T={T} H={H} k={k}")


def test_combine_identity_expert_returns_x_exactly(dev, O):
    """expert_out = expanded_x and renormalised weights: sum_j w_j x rounds
    back to x bit for bit (the weights sum to 1 within k float32 ulps)."""
    from memory_bound_moe_gb300 import moe_combine, moe_expand, moe_route
    for (T, H, E, k) in [(4096, 2048, 128, 8), (1023, 2880, 32, 4), (64, 256, 8, 2)]:
        logits = torch.from_numpy(_logits(T, E, "normal", seed=T)).to(dev)
        x = bf16_dev(_rand_bf16(O, (T, H), seed=k), dev)
        r = moe_route(logits, k, True)
        ex = moe_expand(x, r.inv_perm, k)
        out = moe_combine(ex, r.topk_weights, r.inv_perm)
        torch.cuda.synchronize()
        check_exact(u16(out), u16(x), f"identity T={T}")


def test_out_of_range_indices_are_skipped(dev, O):
    from memory_bound_moe_gb300 import moe_combine, moe_expand
    T, H, k = 8, 64, 2
    x = _rand_bf16(O, (T, H), seed=3)
    inv = np.arange(T * k, dtype=np.int32)
    inv[5] = -1
    inv[6] = T * k + 100
    canary = torch.full((T * k, H), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
    moe_expand(bf16_dev(x, dev), torch.from_numpy(inv).to(dev), k, out=canary)
    got = u16(canary)
    assert np.all(got[6] == 0xFFFF) and np.all(got[5] == 0xFFFF)   # nothing written there
    w = np.ones((T, k), dtype=np.float32)
    eo = _rand_bf16(O, (T * k, H), seed=4)
    out = u16(moe_combine(bf16_dev(eo, dev), torch.from_numpy(w).to(dev), torch.from_numpy(inv).to(dev)))
    inv_ok = inv.copy()
    inv_ok[5] = 0
    inv_ok[6] = 0
    w_ok = w.copy()
    w_ok[2, 1] = 0.0    # slot 5 = token 2, j 1
    w_ok[3, 0] = 0.0    # slot 6 = token 3, j 0
    check_bf16_close(out, O.combine(eo, w_ok, inv_ok), "skipped terms")


def test_parity_check_catches_a_single_flipped_element(dev, O):
    """Negative control: the comparison used above fails on one corrupted
    element (planted in the oracle's result, on the CPU)."""
    from memory_bound_moe_gb300 import moe_swiglu
    w, inp = workload_inputs("tiny")
    gu = u16(inp["gate_up"])
    got = u16(moe_swiglu(bf16_dev(gu, dev)))
    ref = O.swiglu(gu).copy()
    check_bf16_close(got, ref)
    ref[3, 7] ^= 0x4000                      # flip an exponent bit
    with pytest.raises(AssertionError):
        check_bf16_close(got, ref)
    r = O.route(inp["logits"].numpy(), w.k, w.renorm)
    g = gpu_route(dev, inp["logits"].numpy(), w.k, w.renorm)
    bad = dict(r)
    bad["perm"] = r["perm"].copy()
    bad["perm"][[0, 1]] = bad["perm"][[1, 0]]
    with pytest.raises(AssertionError):
        assert_route_equal(g, bad, "planted swap")


# ---------------------------------------------------------------------------
# route + expand in one call (one launch for decode-sized batches)
# ---------------------------------------------------------------------------

ROUTE_EXPAND_CASES = [
    # T, E, k, H, renorm  (the first rows take the one-launch path)
    (1, 8, 2, 64, True), (7, 3, 3, 24, True), (16, 256, 8, 7168, False), (32, 64, 4, 2880, True),
    (64, 8, 2, 256, True), (128, 8, 8, 16, False), (5, 1024, 16, 512, True), (30, 16, 5, 8, True),
    (33, 64, 4, 256, True), (1023, 32, 4, 2880, True),       # two-kernel route + expand
    (4096, 128, 8, 2048, True), (8192, 8, 2, 4096, True), (2000, 1024, 16, 64, False),
    (777, 99, 6, 200, True), (300, 16, 3, 136, False),
]


@pytest.mark.parametrize("T,E,k,H,renorm", ROUTE_EXPAND_CASES)
@pytest.mark.parametrize("wide", [True, False])
def test_route_expand_matches_oracle_and_separate_calls(dev, O, T, E, k, H, renorm, wide):
    from memory_bound_moe_gb300 import moe_expand, moe_route, moe_route_expand
    logits = _logits(T, E, "ties" if T % 2 else "normal", seed=T + E + H)
    x = _rand_bf16(O, (T, H), seed=H + k)
    ld = torch.from_numpy(logits).to(dev)
    xd = bf16_dev(x, dev)
    expanded = torch.full((T * k, H), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
    if not wide:
        xd = _offset16(xd)
        expanded = _offset16(expanded)
    r, ex = moe_route_expand(ld, xd, k, renorm, expanded=expanded)
    torch.cuda.synchronize()
    ref = O.route(logits, k, renorm)
    assert_route_equal({f: getattr(r, f).cpu().numpy() for f in r._fields}, ref, f"T={T} E={E}")
    check_exact(u16(ex), O.expand(x, k, ref["perm"]), f"expanded T={T} E={E} k={k} H={H}")
    # bit-identical to the two separate calls
    r2 = moe_route(ld, k, renorm)
    ex2 = moe_expand(xd, r2.inv_perm, k)
    torch.cuda.synchronize()
    for f in r._fields:
        assert torch.equal(getattr(r, f), getattr(r2, f)), f
    assert torch.equal(ex.view(torch.int16), ex2.view(torch.int16))
