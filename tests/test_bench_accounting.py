"""The benchmark's byte accounting, on CPU.

bench.py reports GB/s and roofline fractions from closed-form algorithmic
bytes per kernel: every input byte read once and every output byte written
once. Here the same figures are rebuilt from the tensors each C-ABI call
reads and writes (shape x element size, as the header declares them), so a
wrong term in a formula (2SH written as 2TH, a missing index array) fails.
The committed ncu DRAM rows are also held to the accounting: no kernel may
move more than its algorithmic bytes (a re-read would show as more).
"""
from __future__ import annotations

import os

import pytest

import bench
from memory_bound_moe_gb300.workloads import WORKLOADS

F32, I32, BF16 = 4, 4, 2


def _tensors(w):
    """Per call: (inputs, outputs) as (rows, cols, element bytes)."""
    T, H, E, k, I, S = w.T, w.H, w.E, w.k, w.I, w.S
    return {
        "route": ([(T, E, F32)],                                         # logits
                  [(T, k, I32), (T, k, F32), (S, 1, I32), (S, 1, I32),   # ids, weights, perm, inv_perm
                   (E, 1, I32), (E + 1, 1, I32)]),                       # counts, offsets
        "expand": ([(T, H, BF16), (S, 1, I32)],                          # x, inv_perm
                   [(S, H, BF16)]),                                      # expanded rows
        "swiglu": ([(S, 2 * I, BF16)],                                   # gate_up
                   [(S, I, BF16)]),                                      # act
        "combine": ([(S, H, BF16), (T, k, F32), (S, 1, I32)],            # expert rows, weights, inv_perm
                    [(T, H, BF16)]),                                     # out
    }


def _nbytes(ts):
    return sum(r * c * b for r, c, b in ts)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_algorithmic_bytes_match_the_calls_tensors(name):
    w = WORKLOADS[name]
    ab = bench.algorithmic_bytes(w)
    tensors = _tensors(w)
    assert set(ab) == set(tensors)
    for kern, (ins, outs) in tensors.items():
        assert ab[kern] == _nbytes(ins) + _nbytes(outs), (name, kern)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_step_inputs_are_the_four_external_tensors(name):
    w = WORKLOADS[name]
    total, inputs = bench.step_bytes(w)
    assert total == sum(bench.algorithmic_bytes(w).values())
    T, H, E, I, S = w.T, w.H, w.E, w.I, w.S
    assert inputs == _nbytes([(T, E, F32), (T, H, BF16), (S, 2 * I, BF16), (S, H, BF16)])


def test_committed_dram_traffic_stays_within_the_algorithmic_bytes():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                        "dram_traffic.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows
    for kern, wl, nbytes, _sha in rows:
        ab = bench.algorithmic_bytes(WORKLOADS[wl])[kern]
        assert int(nbytes) <= ab * 1.01, (kern, wl, int(nbytes), ab)
