"""Every validation error leaves the caller's buffers untouched, on a GPU,
with real device memory.

All buffers of the calls below are regions of one 16 MiB device arena
filled with seeded random bytes. Each call breaks one rule of the C ABI
(misaligned pointer or row, k > E, E or k above the build's limits, a NULL
pointer, overlapping buffers, a workspace too small, a bad NVFP4 tensor
scale, a bad local expert range, an unsupported head size) and must return
its status code.

The calls are first made while their stream is being captured into a CUDA
graph: a launch or a memset that got past the validation would be recorded
as a graph node instead of running, so the graph must come out empty (a
valid call captured the same way does add nodes, the positive control). The
graph is destroyed without ever being instantiated. Only then are the same
calls made on a live stream, after which every byte of the arena must still
hold its random value.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

OK, INVALID, MISALIGNED, UNSUPPORTED, WORKSPACE, CUDA = range(6)
NV, MX = 0, 1

_vp, _sz, _int = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_moe_gb300 import binding, build
    build.build()
    lib = binding.load_library()
    lib.moe_route_static.argtypes = [_vp, ctypes.c_int64, _int, _int, _int] + [_vp] * 6 + [_vp]
    lib.moe_route_static.restype = _int
    rt = None
    with open("/proc/self/maps") as fh:
        for line in fh:
            path = line.split()[-1]
            if "libcudart.so" in os.path.basename(path) and path.startswith("/"):
                rt = ctypes.CDLL(path)
                break
    assert rt is not None, "libcudart not loaded"
    rt.cudaStreamBeginCapture.argtypes = [_vp, _int]
    rt.cudaStreamEndCapture.argtypes = [_vp, ctypes.POINTER(_vp)]
    rt.cudaGraphGetNodes.argtypes = [_vp, _vp, ctypes.POINTER(_sz)]
    rt.cudaGraphDestroy.argtypes = [_vp]
    return lib, rt


class Arena:
    """One device buffer cut into 4 KiB-aligned regions."""

    def __init__(self, nbytes, dev):
        g = torch.Generator(device=dev)
        g.manual_seed(1234)
        self.buf = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev, generator=g)
        self.base = self.buf.data_ptr()
        assert self.base % 256 == 0
        self.used = 0

    def region(self, nbytes):
        p = self.base + self.used
        self.used += (nbytes + 4095) // 4096 * 4096
        assert self.used <= self.buf.numel()
        return p


def _failing_calls(lib, a: Arena):
    """(name, call, expected status): every call breaks exactly one rule."""
    T, E, k, H, I = 64, 16, 4, 256, 256
    S = T * k
    lg = a.region(4 * T * E)
    ids, wts = a.region(4 * S), a.region(4 * S)
    cnt, off = a.region(4 * E), a.region(4 * (E + 1))
    perm, inv = a.region(4 * S), a.region(4 * S)
    x, gu, eo = a.region(2 * T * H), a.region(2 * S * 2 * I), a.region(2 * S * H)
    ex, act, out = a.region(2 * S * H), a.region(2 * S * I), a.region(2 * T * H)
    codes, scales = a.region(S * H), a.region(S * H // 16)
    # a batch that takes the two-kernel routing path and needs a workspace
    T2, E2, k2 = 4096, 128, 8
    S2 = T2 * k2
    need = ctypes.c_size_t(0)
    assert lib.moe_route_workspace_size(T2, E2, k2, ctypes.byref(need)) == OK and need.value > 0
    lg2 = a.region(4 * T2 * E2)
    o2 = [a.region(4 * S2), a.region(4 * S2), a.region(4 * E2), a.region(4 * (E2 + 1)),
          a.region(4 * S2), a.region(4 * S2)]
    ws2 = a.region(need.value)
    q, kk, qw, kw = a.region(2 * T * 8 * 128), a.region(2 * T * 2 * 128), a.region(256), a.region(256)

    def route(T=T, E=E, k=k, lg=lg, ids=ids, wts=wts, cnt=cnt, off=off, perm=perm, inv=inv, ws=0, wsb=0):
        return lambda s: lib.moe_route(lg, T, E, k, 1, ids, wts, cnt, off, perm, inv, ws, wsb, s)

    def route2(ws=ws2, wsb=need.value):
        return lambda s: lib.moe_route(lg2, T2, E2, k2, 1, *o2, ws, wsb, s)

    def local(e0=0, e1=8, pad=16, k=k):
        return lambda s: lib.moe_route_local(lg, T, E, k, 1, e0, e1, pad, ids, wts, cnt, off, perm, inv, 0, 0, s)

    def route_expand(H=H, x=x, ex=ex):
        return lambda s: lib.moe_route_expand(lg, T, E, k, 1, x, H, ids, wts, cnt, off, perm, inv, ex, 0, 0, s)

    c = [
        ("route k > E", route(k=E + 1), INVALID),
        ("route k = 0", route(k=0), INVALID),
        ("route E > 1024", route(E=2000, k=2), UNSUPPORTED),
        ("route k > 16", route(E=16 * 4, k=17), UNSUPPORTED),
        ("route logits misaligned", route(lg=lg + 2), MISALIGNED),
        ("route perm misaligned", route(perm=perm + 2), MISALIGNED),
        ("route perm NULL", route(perm=0), INVALID),
        ("route ids over logits", route(ids=lg + 64), INVALID),
        ("route inv_perm over perm", route(inv=perm + 8), INVALID),
        ("route no workspace", route2(ws=0, wsb=0), WORKSPACE),
        ("route workspace one byte short", route2(wsb=need.value - 1), WORKSPACE),
        ("route workspace misaligned", route2(ws=ws2 + 4), MISALIGNED),
        ("route workspace over logits", route2(ws=lg2), INVALID),
        ("route_static k > E", lambda s: lib.moe_route_static(lg, T, E, E + 1, 1, ids, wts, cnt, off, perm,
                                                             inv, s), INVALID),
        ("route_expand H % 8", route_expand(H=H - 6), MISALIGNED),
        ("route_expand x misaligned", route_expand(x=x + 8), MISALIGNED),
        ("route_expand expanded over logits", route_expand(ex=lg), INVALID),
        ("route_local e0 < 0", local(e0=-1), INVALID),
        ("route_local empty range", local(e0=8, e1=8), INVALID),
        ("route_local pad 0", local(pad=0), INVALID),
        ("expand H % 8", lambda s: lib.moe_expand(x, T, H - 6, k, inv, ex, s), MISALIGNED),
        ("expand x misaligned", lambda s: lib.moe_expand(x + 8, T, H, k, inv, ex, s), MISALIGNED),
        ("expand out over x", lambda s: lib.moe_expand(x, T, H, k, inv, x + 512, s), INVALID),
        ("expand k > 16", lambda s: lib.moe_expand(x, T, H, 17, inv, ex, s), UNSUPPORTED),
        ("expand_rows rows < 0", lambda s: lib.moe_expand_rows(x, T, H, k, inv, -1, ex, s), INVALID),
        ("swiglu I % 8", lambda s: lib.moe_swiglu(gu, S, I - 4, act, s), MISALIGNED),
        ("swiglu gate_up misaligned", lambda s: lib.moe_swiglu(gu + 4, S, I, act, s), MISALIGNED),
        ("swiglu act over gate_up", lambda s: lib.moe_swiglu(gu, S, I, gu + 1024, s), INVALID),
        ("combine out misaligned", lambda s: lib.moe_combine(eo, T, H, k, wts, inv, out + 8, s), MISALIGNED),
        ("combine weights misaligned", lambda s: lib.moe_combine(eo, T, H, k, wts + 2, inv, out, s), MISALIGNED),
        ("combine out over weights", lambda s: lib.moe_combine(eo, T, H, k, wts, inv, wts, s), INVALID),
        ("combine_rows out over expert_out",
         lambda s: lib.moe_combine_rows(eo, S, T, H, k, wts, inv, eo + 512, s), INVALID),
        ("swiglu_mxfp8 I % 32", lambda s: lib.moe_swiglu_mxfp8(gu, S, 48, codes, scales, s), MISALIGNED),
        ("swiglu_mxfp8 codes over gate_up", lambda s: lib.moe_swiglu_mxfp8(gu, S, I, gu + 64, scales, s), INVALID),
        ("expand_mxfp8 codes over x",
         lambda s: lib.moe_expand_mxfp8(x, T, H, k, inv, S, x, scales, s), INVALID),
        ("swiglu_fp4 NVFP4 scale 0", lambda s: lib.moe_swiglu_fp4(gu, S, I, NV, 0.0, codes, scales, s), INVALID),
        ("swiglu_fp4 NVFP4 scale < 0", lambda s: lib.moe_swiglu_fp4(gu, S, I, NV, -1.0, codes, scales, s), INVALID),
        ("swiglu_fp4 NVFP4 scale inf",
         lambda s: lib.moe_swiglu_fp4(gu, S, I, NV, math.inf, codes, scales, s), INVALID),
        ("swiglu_fp4 NVFP4 scale nan",
         lambda s: lib.moe_swiglu_fp4(gu, S, I, NV, math.nan, codes, scales, s), INVALID),
        ("swiglu_fp4 unknown format", lambda s: lib.moe_swiglu_fp4(gu, S, I, 2, 1.0, codes, scales, s), INVALID),
        ("swiglu_fp4 NVFP4 I % 16", lambda s: lib.moe_swiglu_fp4(gu, S, 40, NV, 1.0, codes, scales, s), MISALIGNED),
        ("expand_fp4 MXFP4 H % 32",
         lambda s: lib.moe_expand_fp4(x, T, 264, k, inv, S, MX, 0.0, codes, scales, s), MISALIGNED),
        ("expand_fp4 NVFP4 scale NULL",
         lambda s: lib.moe_expand_fp4(x, T, H, k, inv, S, NV, 1.0, codes, 0, s), INVALID),
        ("qk_rmsnorm head_dim 96", lambda s: lib.moe_qk_rmsnorm(q, kk, T, 8, 2, 96, qw, kw, 0.0, 1e-6, s),
         UNSUPPORTED),
        ("qk_rmsnorm q misaligned", lambda s: lib.moe_qk_rmsnorm(q + 8, kk, T, 8, 2, 128, qw, kw, 0.0, 1e-6, s),
         MISALIGNED),
        ("qk_rmsnorm weight inside q", lambda s: lib.moe_qk_rmsnorm(q, kk, T, 8, 2, 128, q + 256, kw, 0.0, 1e-6, s),
         INVALID),
    ]
    valid = lambda s: lib.moe_swiglu(gu, S, I, act, s)       # the positive control
    return c, valid


def _captured_nodes(rt, stream, fn):
    """Call fn(stream) while the stream is captured (relaxed mode); return
    (fn's result, number of nodes in the captured graph). The graph is
    destroyed, never instantiated, so nothing captured ever runs."""
    assert rt.cudaStreamBeginCapture(stream, 2) == 0
    try:
        res = fn(stream)
    finally:
        graph = _vp()
        err = rt.cudaStreamEndCapture(stream, ctypes.byref(graph))
    assert err == 0, err
    n = _sz(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    assert rt.cudaGraphDestroy(graph) == 0
    return res, n.value


def test_every_error_leaves_outputs_untouched(env):
    lib, rt = env
    dev = torch.device("cuda:0")
    arena = Arena(16 << 20, dev)
    calls, valid = _failing_calls(lib, arena)
    torch.cuda.synchronize(dev)
    before = arena.buf.cpu()
    side = torch.cuda.Stream(dev)
    sp = side.cuda_stream

    # positive control: a valid call under capture records its launch
    assert valid(sp) == OK                     # first call outside capture (warms the launch caches)
    torch.cuda.synchronize(dev)
    before = arena.buf.cpu()                   # the valid call wrote act; take the reference after it
    st, n = _captured_nodes(rt, sp, valid)
    assert st == OK and n >= 1, (st, n)

    # every failing call: its status, and nothing enqueued
    for name, fn, want in calls:
        st, n = _captured_nodes(rt, sp, fn)
        assert st == want, (name, st, want)
        assert n == 0, (name, n)

    # the same calls on the live stream, then every byte of the arena
    for name, fn, want in calls:
        assert fn(sp) == want, name
    torch.cuda.synchronize(dev)
    after = arena.buf.cpu()
    diff = torch.nonzero(after != before)
    assert diff.numel() == 0, f"{diff.shape[0]} bytes changed, first at {diff[:5].flatten().tolist()}"
