"""Local (one tensor-parallel rank's) routing with padded expert segments,
expansion into the padded buffer and the partial combine, on the GPU through
the C ABI, against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import bf16_bits_to_f64, check_bf16_close, check_exact, check_weights_close

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


def _logits(T, E, seed, hot=0):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[:, :hot] += 3.0
    return l


LOCAL_CASES = [
    # T, E, k, renorm, e0, e1, pad, hot
    (4096, 128, 8, True, 32, 64, 128, 0),     # two-kernel path, GEMM-tile padding
    (8192, 8, 2, True, 2, 4, 64, 0),
    (16, 256, 8, False, 0, 64, 16, 0),        # one-block path
    (1023, 32, 4, True, 0, 4, 1, 4),          # hot experts, no padding
    (64, 8, 2, True, 7, 8, 3, 0),             # one-block path, 8-lane groups
    (300, 1024, 16, True, 1000, 1024, 8, 0),  # 32 experts per lane
    (5000, 64, 4, True, 10, 11, 256, 0),      # a single local expert
]


@pytest.mark.parametrize("T,E,k,renorm,e0,e1,pad,hot", LOCAL_CASES)
def test_route_local_matches_oracle(dev, oracle_mod, T, E, k, renorm, e0, e1, pad, hot):
    from memory_bound_moe_gb300 import moe_route_local
    O = oracle_mod
    logits = _logits(T, E, T + e0, hot)
    r = moe_route_local(torch.from_numpy(logits).to(dev), k, renorm, e0, e1, pad)
    torch.cuda.synchronize()
    ids, w = O.route_topk(logits, k, renorm)
    counts, offsets, perm, inv = O.route_permute_local(ids, E, e0, e1, pad)
    what = f"T={T} E={E} [{e0},{e1}) pad={pad}"
    check_exact(r.topk_ids.cpu().numpy(), ids, what + " ids")
    check_weights_close(r.topk_weights.cpu().numpy(), w, what + " weights")
    check_exact(r.expert_counts.cpu().numpy(), counts, what + " counts")
    check_exact(r.expert_offsets.cpu().numpy(), offsets, what + " offsets")
    check_exact(r.perm.cpu().numpy(), perm, what + " perm")
    check_exact(r.inv_perm.cpu().numpy(), inv, what + " inv_perm")


@pytest.mark.parametrize("T,E,k", [(4096, 128, 8), (16, 256, 8), (1023, 32, 4)])
def test_route_local_full_range_equals_route(dev, T, E, k):
    from memory_bound_moe_gb300 import moe_route, moe_route_local
    logits = torch.from_numpy(_logits(T, E, 5)).to(dev)
    a = moe_route(logits, k, True)
    b = moe_route_local(logits, k, True, 0, E, 1)
    torch.cuda.synchronize()
    for f in a._fields:
        assert torch.equal(getattr(a, f), getattr(b, f)), f


@pytest.mark.parametrize("T,H,E,k,pad", [(4096, 2048, 128, 8, 128), (1023, 2880, 32, 4, 64),
                                          (16, 7168, 256, 8, 16)])
def test_ranks_expand_and_partial_combines(dev, oracle_mod, T, H, E, k, pad):
    """Four ranks of the experts: each expands into its padded buffer and
    combines its partial sum; the partials add up to the full combine."""
    from memory_bound_moe_gb300 import moe_combine_rows, moe_expand_rows, moe_route_local
    O = oracle_mod
    rng = np.random.default_rng(T + H)
    logits = _logits(T, E, T)
    x = O.bf16_round(rng.standard_normal((T, H)))
    eo_full = O.bf16_round(rng.standard_normal((T * k, H)))   # expert outputs per global slot row
    full = O.route(logits, k, True)
    ld, xd = torch.from_numpy(logits).to(dev), bf16_dev(x, dev)
    total = np.zeros((T, H))
    mag = np.zeros((T, H))
    bounds = np.linspace(0, E, 5).astype(int)
    for e0, e1 in zip(bounds[:-1], bounds[1:]):
        r = moe_route_local(ld, k, True, int(e0), int(e1), pad)
        rows = r.perm.numel()
        canary = torch.full((rows, H), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
        ex = moe_expand_rows(xd, r.inv_perm, k, rows, out=canary)
        torch.cuda.synchronize()
        perm = r.perm.cpu().numpy()
        ref = np.full((rows, H), 0xFFFF, dtype=np.uint16)
        O.expand_into(x, k, perm, ref)            # padding rows keep the canary
        check_exact(u16(ex), ref, f"expanded rank [{e0},{e1})")
        # this rank's expert outputs: the full slot rows placed at its rows
        eo = np.zeros((rows, H), dtype=np.uint16)
        valid = perm >= 0
        eo[valid] = eo_full[full["inv_perm"][perm[valid]]]
        part = moe_combine_rows(bf16_dev(eo, dev), r.topk_weights, r.inv_perm)
        ref_part = O.combine(eo, full["topk_weights"], r.inv_perm.cpu().numpy())
        check_bf16_close(u16(part), ref_part, f"partial combine [{e0},{e1})")
        total += bf16_bits_to_f64(u16(part))
        mag += np.abs(bf16_bits_to_f64(u16(part)))
    ref_full = bf16_bits_to_f64(O.combine(eo_full, full["topk_weights"], full["inv_perm"]))
    # the simulated all-reduce: every partial rounded once, then summed
    err = np.abs(total - ref_full)
    assert np.all(err <= 2e-2 + 2 ** -7 * (mag + np.abs(ref_full))), float(err.max())


def test_route_local_empty_batch(dev):
    from memory_bound_moe_gb300 import moe_route_local
    r = moe_route_local(torch.empty((0, 64), dtype=torch.float32, device=dev), 4, True, 8, 24, 4)
    torch.cuda.synchronize()
    assert r.expert_counts.cpu().tolist() == [0] * 16
    assert r.expert_offsets.cpu().tolist() == [0] * 17
    assert r.perm.numel() == 16 * 3 and bool((r.perm == -1).all())
