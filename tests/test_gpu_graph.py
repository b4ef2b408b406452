"""One MoE layer captured into a CUDA graph.

Every kernel of the library is launched with programmatic stream
serialisation (programmatic dependent launch). Captured from a stream, the
four calls of a decode layer (route, expand, SwiGLU, combine) must become
four kernel nodes joined by programmatic edges, so that a replayed graph
keeps the launch overlap of the stream. The replayed graph's outputs must
be bit-identical to the same calls launched on the stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

_vp, _sz, _int, _ull = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_ulonglong


class EdgeData(ctypes.Structure):
    _fields_ = [("from_port", ctypes.c_ubyte), ("to_port", ctypes.c_ubyte), ("type", ctypes.c_ubyte),
                ("reserved", ctypes.c_ubyte * 5)]


PROGRAMMATIC = 1   # cudaGraphDependencyTypeProgrammatic


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_moe_gb300 import binding, build
    build.build()
    lib = binding.load_library()
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
    rt.cudaGraphGetEdges.argtypes = [_vp, _vp, _vp, _vp, ctypes.POINTER(_sz)]
    rt.cudaGraphInstantiate.argtypes = [ctypes.POINTER(_vp), _vp, _ull]
    rt.cudaGraphLaunch.argtypes = [_vp, _vp]
    rt.cudaGraphExecDestroy.argtypes = [_vp]
    rt.cudaGraphDestroy.argtypes = [_vp]
    return lib, rt


def test_decode_layer_graph_keeps_programmatic_edges(env):
    lib, rt = env
    from memory_bound_moe_gb300.workloads import WORKLOADS, generate
    dev = torch.device("cuda:0")
    w = WORKLOADS["decode"]
    inp = {k: v.to(dev) for k, v in generate(w, seed=3).items()}
    T, E, k, S, H, I = w.T, w.E, w.k, w.S, w.H, w.I
    i32 = dict(dtype=torch.int32, device=dev)

    def buffers():
        return {"ids": torch.empty((T, k), **i32), "w": torch.empty((T, k), dtype=torch.float32, device=dev),
                "cnt": torch.empty((E,), **i32), "off": torch.empty((E + 1,), **i32),
                "perm": torch.empty((S,), **i32), "inv": torch.empty((S,), **i32),
                "ex": torch.empty((S, H), dtype=torch.bfloat16, device=dev),
                "act": torch.empty((S, I), dtype=torch.bfloat16, device=dev),
                "out": torch.empty((T, H), dtype=torch.bfloat16, device=dev)}

    p = lambda t: t.data_ptr()

    def layer(b, sp):
        st = lib.moe_route(p(inp["logits"]), T, E, k, int(w.renorm), p(b["ids"]), p(b["w"]), p(b["cnt"]),
                           p(b["off"]), p(b["perm"]), p(b["inv"]), 0, 0, sp)
        st |= lib.moe_expand(p(inp["x"]), T, H, k, p(b["inv"]), p(b["ex"]), sp)
        st |= lib.moe_swiglu(p(inp["gate_up"]), S, I, p(b["act"]), sp)
        st |= lib.moe_combine(p(inp["expert_out"]), T, H, k, p(b["w"]), p(b["inv"]), p(b["out"]), sp)
        assert st == 0

    side = torch.cuda.Stream(dev)
    sp = side.cuda_stream
    ref, got = buffers(), buffers()
    layer(ref, sp)                        # stream launch (also loads every kernel before capture)
    torch.cuda.synchronize(dev)

    assert rt.cudaStreamBeginCapture(sp, 2) == 0     # relaxed
    try:
        layer(got, sp)
    finally:
        graph = _vp()
        err = rt.cudaStreamEndCapture(sp, ctypes.byref(graph))
    assert err == 0
    try:
        n = _sz(0)
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        assert n.value == 4, n.value                 # one kernel per call (decode routes in one block)
        ne = _sz(0)
        assert rt.cudaGraphGetEdges(graph, None, None, None, ctypes.byref(ne)) == 0
        frm, to = (_vp * max(ne.value, 1))(), (_vp * max(ne.value, 1))()
        data = (EdgeData * max(ne.value, 1))()
        assert rt.cudaGraphGetEdges(graph, frm, to, data, ctypes.byref(ne)) == 0
        types = [data[i].type for i in range(ne.value)]
        assert ne.value == 3, types                  # a chain of the four kernels
        assert all(t == PROGRAMMATIC for t in types), types
        exe = _vp()
        assert rt.cudaGraphInstantiate(ctypes.byref(exe), graph, 0) == 0
        try:
            for _ in range(3):                       # replays write the same outputs
                assert rt.cudaGraphLaunch(exe, sp) == 0
            torch.cuda.synchronize(dev)
        finally:
            assert rt.cudaGraphExecDestroy(exe) == 0
    finally:
        assert rt.cudaGraphDestroy(graph) == 0
    for name in ref:
        assert torch.equal(ref[name].view(torch.uint8) if ref[name].dtype == torch.bfloat16 else ref[name],
                           got[name].view(torch.uint8) if got[name].dtype == torch.bfloat16 else got[name]), name
