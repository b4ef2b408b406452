"""moe_route_static, the routing entry point that allocates nothing.

It exists for callers that may not allocate device memory where they route
(a runtime that owns all device memory from start-up, an allocator-free
host, a call site that cannot afford cudaMalloc's possible synchronisation):
its scratch is a fixed 128 KiB device array inside the library instead of a
caller workspace.

* Two calls in a row through the C ABI, with different shapes that both use
  the scratch, each checked against moe_route on the same inputs and against
  the oracle's routing.
* A child process calls it, resets the device (cudaDeviceReset, which ends
  that process's CUDA context and unloads the library's device code), and
  calls it again: the second call must find the array in the new context.

The file runs last so that a failure here leaves the rest of the suite
already run, and it passes alone in a fresh process too.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from helpers import check_exact, check_weights_close

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _lib():
    from memory_bound_moe_gb300 import binding, build
    build.build()
    lib = binding.load_library()
    f = lib.moe_route_static
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int] + \
                 [ctypes.c_void_p] * 6 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


FIELDS = ("topk_ids", "topk_weights", "expert_counts", "expert_offsets", "perm", "inv_perm")


def _assert_route(got, ref, what):
    for f in FIELDS:
        if f == "topk_weights":
            check_weights_close(got[f], ref[f], f"{what} weights")
        else:
            check_exact(got[f], ref[f], f"{what} {f}")


def test_static_scratch_route_matches_workspace_route(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_moe_gb300 import moe_route, moe_route_workspace_size
    lib = _lib()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    # two calls in a row; both shapes take the two-kernel path, so both use
    # the static scratch, and the second must not be disturbed by what the
    # first left in it
    cases = [(4096, 128, 8, True, 11), (1023, 32, 4, False, 12)]
    for T, E, k, renorm, seed in cases:
        assert 0 < moe_route_workspace_size(T, E, k) <= 128 * 1024
        rng = np.random.default_rng(seed)
        logits_np = rng.standard_normal((T, E)).astype(np.float32)
        logits = torch.from_numpy(logits_np).to(dev)
        ref = moe_route(logits, k, renorm)
        i32 = dict(dtype=torch.int32, device=dev)
        ids = torch.empty((T, k), **i32)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        counts = torch.empty((E,), **i32)
        offsets = torch.empty((E + 1,), **i32)
        perm = torch.empty((T * k,), **i32)
        inv = torch.empty((T * k,), **i32)
        st = lib.moe_route_static(logits.data_ptr(), T, E, k, int(renorm), ids.data_ptr(),
                                  w.data_ptr(), counts.data_ptr(), offsets.data_ptr(),
                                  perm.data_ptr(), inv.data_ptr(), stream.cuda_stream)
        assert st == 0, st
        torch.cuda.synchronize(dev)
        got = {"topk_ids": ids, "topk_weights": w, "expert_counts": counts, "expert_offsets": offsets,
               "perm": perm, "inv_perm": inv}
        got = {f: v.cpu().numpy() for f, v in got.items()}
        what = f"T={T} E={E} k={k}"
        _assert_route(got, {f: getattr(ref, f).cpu().numpy() for f in FIELDS}, f"{what} vs moe_route")
        _assert_route(got, oracle_mod.route(logits_np, k, renorm), f"{what} vs oracle")


def test_static_scratch_route_after_device_reset(oracle_mod, tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib()                                         # built in-tree before the child loads it
    T, E, k, renorm, seed = 4096, 128, 8, 1, 21
    out = tmp_path / "reset.npz"
    res = subprocess.run([sys.executable, os.path.join(HERE, "static_route_reset_child.py"), str(out),
                          str(T), str(E), str(k), str(renorm), str(seed)],
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-2000:]
    d = np.load(out)
    ref = oracle_mod.route(d["logits"], k, bool(renorm))
    for call in (0, 1):
        _assert_route({f: d[f"{f}{call}"] for f in FIELDS}, ref, f"call {call}")
