"""moe_route_static, the routing entry point that allocates nothing.

It exists for callers that may not allocate device memory where they route
(a runtime that owns all device memory from start-up, an allocator-free
host, a call site that cannot afford cudaMalloc's possible synchronisation):
its scratch is a fixed 128 KiB device array inside the library instead of a
caller workspace. This test calls it through the C ABI twice in a row, with
different shapes that both use the scratch, and checks each result against
moe_route on the same inputs. It runs last so that a failure here leaves the
rest of the suite already run, and it passes alone in a fresh process too.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from helpers import check_exact, check_weights_close

pytestmark = pytest.mark.gpu


def _lib():
    from memory_bound_moe_gb300 import binding, build
    build.build()
    lib = binding.load_library()
    f = lib.moe_route_static
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int] + \
                 [ctypes.c_void_p] * 6 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def test_static_scratch_route_matches_workspace_route():
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
        logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).to(dev)
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
        what = f"T={T} E={E} k={k}"
        check_exact(ids.cpu().numpy(), ref.topk_ids.cpu().numpy(), f"{what} ids")
        check_exact(counts.cpu().numpy(), ref.expert_counts.cpu().numpy(), f"{what} counts")
        check_exact(offsets.cpu().numpy(), ref.expert_offsets.cpu().numpy(), f"{what} offsets")
        check_exact(perm.cpu().numpy(), ref.perm.cpu().numpy(), f"{what} perm")
        check_exact(inv.cpu().numpy(), ref.inv_perm.cpu().numpy(), f"{what} inv_perm")
        check_weights_close(w.cpu().numpy(), ref.topk_weights.cpu().numpy(), f"{what} weights")
