"""The C-ABI library without a GPU: it loads, exports every function that
``include/*.h`` declares, and its host-side validation rejects bad arguments
before any CUDA call (only fake, never-dereferenced addresses are passed, and
every call here returns before a launch)."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

OK, INVALID, MISALIGNED, UNSUPPORTED, WORKSPACE, CUDA = range(6)


@pytest.fixture(scope="module")
def lib():
    from memory_bound_moe_gb300 import build as b
    b.build()
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    from memory_bound_moe_gb300 import binding
    return binding.load_library()


@pytest.fixture(scope="module")
def nogpu():
    # The validation tests pass fake device addresses that are never
    # dereferenced because every call fails validation first; on a machine
    # with a GPU they are skipped anyway, so no slip in a test can ever launch
    # a kernel on such an address.
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake-address validation tests run only on hosts without a GPU")


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"moe_route", "moe_expand", "moe_swiglu", "moe_combine",
            "moe_route_workspace_size", "moe_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code, name in enumerate(["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_MISALIGNED",
                                 "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE", "MOE_ERR_CUDA"]):
        assert lib.moe_status_string(code).decode() == name
    assert lib.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"


def _ws(lib, T, E, k):
    out = ctypes.c_size_t(12345)
    st = lib.moe_route_workspace_size(T, E, k, ctypes.byref(out))
    return st, out.value


def test_workspace_size_rules(lib):
    assert _ws(lib, 0, 8, 2) == (OK, 0)
    assert _ws(lib, 16, 256, 8) == (OK, 0)          # one-block path: no workspace
    st, b = _ws(lib, 4096, 128, 8)
    assert st == OK and b > 0 and b % 16 == 0
    st2, b2 = _ws(lib, 4096, 128, 8)
    assert (st2, b2) == (st, b)                       # pure function
    assert _ws(lib, 8192, 8, 2)[0] == OK
    assert _ws(lib, -1, 8, 2)[0] == INVALID
    assert _ws(lib, 10, 8, 9)[0] == INVALID           # k > E
    assert _ws(lib, 10, 8, 0)[0] == INVALID
    assert _ws(lib, 10, 2048, 8)[0] == UNSUPPORTED    # E > 1024
    assert _ws(lib, 10, 64, 17)[0] == UNSUPPORTED     # k > 16
    assert _ws(lib, 2 ** 31 // 4, 64, 4)[0] == UNSUPPORTED
    assert lib.moe_route_workspace_size(10, 8, 2, None) == INVALID


# Fake device addresses, far apart and 256-byte aligned; never dereferenced.
A = [0x7f0000000000 + i * 0x100000000 for i in range(16)]


def _route(lib, T=64, E=8, k=2, ptrs=None, ws=0, ws_bytes=0):
    p = list(A[:7]) if ptrs is None else ptrs
    return lib.moe_route(p[0], T, E, k, 1, p[1], p[2], p[3], p[4], p[5], p[6], ws, ws_bytes, None)


def test_route_rejects_bad_arguments(lib, nogpu):
    assert _route(lib, k=9) == INVALID
    assert _route(lib, k=0) == INVALID
    assert _route(lib, T=-3) == INVALID
    assert _route(lib, E=2000, k=2) == UNSUPPORTED
    assert _route(lib, E=64, k=20) == UNSUPPORTED
    for i in range(7):
        p = list(A[:7])
        p[i] = 0
        assert _route(lib, ptrs=p) == INVALID, i
        p = list(A[:7])
        p[i] += 2                                     # not 4-byte aligned
        assert _route(lib, ptrs=p) == MISALIGNED, i
    # two-kernel path needs a workspace
    st, need = _ws(lib, 4096, 128, 8)
    assert _route(lib, T=4096, E=128, k=8) == WORKSPACE
    assert _route(lib, T=4096, E=128, k=8, ws=A[8], ws_bytes=need - 1) == WORKSPACE
    assert _route(lib, T=4096, E=128, k=8, ws=A[8] + 4, ws_bytes=need) == MISALIGNED
    # outputs overlapping the logits or each other
    p = list(A[:7])
    p[1] = A[0] + 64
    assert _route(lib, ptrs=p) == INVALID
    p = list(A[:7])
    p[6] = p[5] + 8
    assert _route(lib, ptrs=p) == INVALID


def test_expand_swiglu_combine_reject_bad_arguments(lib, nogpu):
    # expand(x, T, H, k, inv_perm, out, stream)
    assert lib.moe_expand(A[0], 16, 256, 0, A[1], A[2], None) == INVALID
    assert lib.moe_expand(A[0], 16, 256, 17, A[1], A[2], None) == UNSUPPORTED
    assert lib.moe_expand(A[0], 16, 250, 2, A[1], A[2], None) == MISALIGNED   # H % 8
    assert lib.moe_expand(A[0] + 8, 16, 256, 2, A[1], A[2], None) == MISALIGNED
    assert lib.moe_expand(A[0], 16, 256, 2, A[1] + 1, A[2], None) == MISALIGNED
    assert lib.moe_expand(0, 16, 256, 2, A[1], A[2], None) == INVALID
    assert lib.moe_expand(A[0], -1, 256, 2, A[1], A[2], None) == INVALID
    assert lib.moe_expand(A[0], 16, 256, 2, A[1], A[0] + 256, None) == INVALID  # out over x
    assert lib.moe_expand(0, 0, 256, 2, 0, 0, None) == OK                       # empty batch
    # swiglu(gate_up, rows, I, act, stream)
    assert lib.moe_swiglu(A[0], 16, 100, A[1], None) == MISALIGNED             # I % 8
    assert lib.moe_swiglu(A[0], 16, 0, A[1], None) == INVALID
    assert lib.moe_swiglu(A[0] + 4, 16, 128, A[1], None) == MISALIGNED
    assert lib.moe_swiglu(A[0], 16, 128, 0, None) == INVALID
    assert lib.moe_swiglu(A[0], 16, 128, A[0] + 1024, None) == INVALID         # act over gate_up
    assert lib.moe_swiglu(0, 0, 128, 0, None) == OK
    # combine(expert_out, T, H, k, w, inv_perm, out, stream)
    assert lib.moe_combine(A[0], 16, 256, 2, A[1], A[2], A[3] + 8, None) == MISALIGNED
    assert lib.moe_combine(A[0], 16, 256, 2, A[1] + 2, A[2], A[3], None) == MISALIGNED
    assert lib.moe_combine(A[0], 16, 256, 2, 0, A[2], A[3], None) == INVALID
    assert lib.moe_combine(A[0], 16, 264, 0, A[1], A[2], A[3], None) == INVALID
    assert lib.moe_combine(A[0], 16, 260, 2, A[1], A[2], A[3], None) == MISALIGNED
    assert lib.moe_combine(A[0], 16, 256, 2, A[1], A[2], A[1], None) == INVALID  # out over w
    assert lib.moe_combine(0, 0, 256, 2, 0, 0, 0, None) == OK


def test_route_expand_rejects_bad_arguments(lib, nogpu):
    def call(T=16, E=64, k=4, H=256, x=A[7], ex=A[8], ws=0, ws_bytes=0, p=None):
        p = list(A[:7]) if p is None else p
        return lib.moe_route_expand(p[0], T, E, k, 1, x, H, p[1], p[2], p[3], p[4], p[5], p[6],
                                    ex, ws, ws_bytes, None)
    assert call(H=250) == MISALIGNED                       # H % 8
    assert call(x=A[7] + 8) == MISALIGNED                  # bf16 rows need 16-byte alignment
    assert call(ex=0) == INVALID
    assert call(x=0) == INVALID
    assert call(k=0) == INVALID
    assert call(E=2000) == UNSUPPORTED
    assert call(ex=A[0]) == INVALID                        # expanded_x over the logits
    assert call(x=A[1]) == INVALID                         # an output over x
    assert call(T=4096, E=128, k=8) == WORKSPACE           # two-kernel path without workspace
    p = list(A[:7])
    p[3] = 0
    assert call(p=p) == INVALID


def test_local_routing_rules(lib, nogpu):
    rows = ctypes.c_int64(0)
    assert lib.moe_route_local_rows(100, 8, 16, 32, 128, ctypes.byref(rows)) == OK
    assert rows.value == 100 * 8 + 16 * 127
    assert lib.moe_route_local_rows(100, 8, 32, 32, 1, ctypes.byref(rows)) == INVALID   # empty range
    assert lib.moe_route_local_rows(100, 8, 0, 4, 0, ctypes.byref(rows)) == INVALID     # pad < 1
    ws = ctypes.c_size_t(0)
    assert lib.moe_route_local_workspace_size(4096, 128, 8, 0, 32, ctypes.byref(ws)) == OK
    full = ctypes.c_size_t(0)
    assert lib.moe_route_workspace_size(4096, 128, 8, ctypes.byref(full)) == OK
    assert 0 < ws.value <= full.value            # narrower count matrix
    assert lib.moe_route_local_workspace_size(4096, 128, 8, 0, 129, ctypes.byref(ws)) == INVALID

    def call(e0=0, e1=32, pad=16, T=16, E=64, k=4, p=None):
        p = list(A[:7]) if p is None else p
        return lib.moe_route_local(p[0], T, E, k, 1, e0, e1, pad, p[1], p[2], p[3], p[4], p[5], p[6],
                                   0, 0, None)
    assert call(e0=-1) == INVALID
    assert call(e1=65) == INVALID
    assert call(e0=10, e1=10) == INVALID
    assert call(pad=0) == INVALID
    assert call(T=4096, E=128, k=8) == WORKSPACE
    p = list(A[:7])
    p[5] = p[0] + 4                               # perm over the logits
    assert call(p=p) == INVALID
    # rows-bounded expand / combine
    assert lib.moe_expand_rows(A[0], 16, 256, 2, A[1], -1, A[2], None) == INVALID
    assert lib.moe_expand_rows(A[0], 16, 250, 2, A[1], 40, A[2], None) == MISALIGNED
    assert lib.moe_combine_rows(A[0], 40, 16, 256, 2, A[1], A[2], A[0] + 512, None) == INVALID
    assert lib.moe_combine_rows(A[0], -3, 16, 256, 2, A[1], A[2], A[3], None) == INVALID


def test_mxfp8_rules(lib, nogpu):
    assert lib.moe_swiglu_mxfp8(A[0], 16, 48, A[1], A[2], None) == MISALIGNED     # I % 32
    assert lib.moe_swiglu_mxfp8(A[0], 16, 64, A[1] + 8, A[2], None) == MISALIGNED  # codes alignment
    assert lib.moe_swiglu_mxfp8(A[0], 16, 64, 0, A[2], None) == INVALID
    assert lib.moe_swiglu_mxfp8(A[0], 16, 64, A[0] + 64, A[2], None) == INVALID   # codes over gate_up
    assert lib.moe_swiglu_mxfp8(0, 0, 64, 0, 0, None) == OK
    assert lib.moe_expand_mxfp8(A[0], 16, 264, 2, A[1], 32, A[2], A[3], None) == MISALIGNED  # H % 32
    assert lib.moe_expand_mxfp8(A[0], 16, 256, 2, A[1], -1, A[2], A[3], None) == INVALID
    assert lib.moe_expand_mxfp8(A[0], 16, 256, 2, A[1], 32, A[2], 0, None) == INVALID
    assert lib.moe_expand_mxfp8(A[0], 16, 256, 2, A[1], 32, A[0], A[3], None) == INVALID   # codes over x


def test_fp4_rules(lib, nogpu):
    NV, MX = 0, 1
    sw = lambda *a: lib.moe_swiglu_fp4(*a)
    assert sw(A[0], 16, 64, 2, 1.0, A[1], A[2], None) == INVALID                  # unknown format
    assert sw(A[0], 16, 64, NV, 0.0, A[1], A[2], None) == INVALID                 # NVFP4 scale must be > 0
    assert sw(A[0], 16, 64, NV, -1.0, A[1], A[2], None) == INVALID
    assert sw(A[0], 16, 64, NV, float("inf"), A[1], A[2], None) == INVALID
    assert sw(A[0], 16, 64, NV, float("nan"), A[1], A[2], None) == INVALID
    assert sw(A[0], 16, 48, MX, 1.0, A[1], A[2], None) == MISALIGNED              # I % 32 for MXFP4
    assert sw(A[0], 16, 40, NV, 1.0, A[1], A[2], None) == MISALIGNED              # I % 16 for NVFP4
    assert sw(A[0], 16, 64, MX, 0.0, A[1] + 8, A[2], None) == MISALIGNED          # codes alignment
    assert sw(A[0], 16, 64, MX, 0.0, 0, A[2], None) == INVALID
    assert sw(A[0], 16, 64, NV, 1.0, A[0] + 64, A[2], None) == INVALID            # codes over gate_up
    assert sw(0, 0, 64, NV, 1.0, 0, 0, None) == OK                                # nothing to do
    ex = lambda *a: lib.moe_expand_fp4(*a)
    assert ex(A[0], 16, 264, 2, A[1], 32, MX, 0.0, A[2], A[3], None) == MISALIGNED   # H % 32
    assert ex(A[0], 16, 264, 2, A[1], 32, NV, 1.0, A[2], A[3], None) == MISALIGNED   # H % 16
    assert ex(A[0], 16, 256, 2, A[1], 32, 5, 1.0, A[2], A[3], None) == INVALID
    assert ex(A[0], 16, 256, 2, A[1], -1, NV, 1.0, A[2], A[3], None) == INVALID
    assert ex(A[0], 16, 256, 2, A[1], 32, NV, 1.0, A[2], 0, None) == INVALID
    assert ex(A[0], 16, 256, 2, A[1], 32, NV, 1.0, A[0], A[3], None) == INVALID      # codes over x
    assert ex(A[0], 16, 256, 17, A[1], 32, NV, 1.0, A[2], A[3], None) == UNSUPPORTED  # k > 16


def test_qk_rmsnorm_rules(lib, nogpu):
    f = lambda *a: lib.moe_qk_rmsnorm(*a)
    import ctypes as C
    lib.moe_qk_rmsnorm.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int, C.c_int, C.c_int,
                                   C.c_void_p, C.c_void_p, C.c_float, C.c_float, C.c_void_p]
    assert f(A[0], A[1], 16, 32, 4, 96, A[2], A[3], 0.0, 1e-6, None) == UNSUPPORTED   # head_dim
    assert f(A[0], A[1], 16, 0, 0, 128, A[2], A[3], 0.0, 1e-6, None) == INVALID
    assert f(A[0] + 8, A[1], 16, 32, 4, 128, A[2], A[3], 0.0, 1e-6, None) == MISALIGNED
    assert f(A[0], A[1], 16, 32, 4, 128, A[2] + 2, A[3], 0.0, 1e-6, None) == MISALIGNED
    assert f(A[0], A[1], 16, 32, 4, 128, A[0] + 256, A[3], 0.0, 1e-6, None) == INVALID  # weight in q
    assert f(0, 0, 0, 32, 4, 128, A[2], A[3], 0.0, 1e-6, None) == OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from memory_bound_moe_gb300 import moe_swiglu
    with pytest.raises(ValueError):
        moe_swiglu(torch.zeros((4, 16), dtype=torch.bfloat16))


def test_product_path_never_imports_the_oracle():
    # the oracle is test infrastructure: nothing in the package loads or calls it
    pat = re.compile(r"\b(import|from)\s+oracle\b|\boracle\.\w+\(|moe_oracle|liboracle|\boracle_\w+\(")
    pkg = os.path.join(ROOT, "memory_bound_moe_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            assert not pat.search(open(path).read()), path
