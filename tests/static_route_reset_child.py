"""Child process of tests/test_zz_no_alloc.py: moe_route_static called once,
then again after cudaDeviceReset, in a process of its own.

Device memory comes straight from the CUDA runtime (cudaMalloc/cudaMemcpy
through ctypes), not from PyTorch: a reset ends the process's CUDA context
and frees every allocation in it, which PyTorch's caching allocator would
not know about. The reset also unloads the library's device code; the
second call must find its static scratch array in the new context.

Usage: python static_route_reset_child.py OUT.npz T E k renorm seed
Writes the outputs of both calls (suffixes 0 and 1) and the logits.
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

_vp, _i64, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
H2D, D2H = 1, 2


def _loaded_cudart():
    """The CUDA runtime the library was linked against (already mapped into
    this process by loading the library)."""
    with open("/proc/self/maps") as fh:
        for line in fh:
            path = line.split()[-1]
            if "libcudart.so" in os.path.basename(path):
                return ctypes.CDLL(path)
    raise RuntimeError("libcudart is not loaded")


def main():
    out_path = sys.argv[1]
    T, E, k, renorm, seed = (int(v) for v in sys.argv[2:7])
    lib = ctypes.CDLL(os.path.join(ROOT, "memory_bound_moe_gb300", "lib", "libmoeglue.so"))
    lib.moe_route_static.argtypes = [_vp, _i64, _int, _int, _int] + [_vp] * 6 + [_vp]
    lib.moe_route_static.restype = _int
    rt = _loaded_cudart()
    rt.cudaSetDevice.argtypes = [_int]
    rt.cudaMalloc.argtypes = [ctypes.POINTER(_vp), _sz]
    rt.cudaFree.argtypes = [_vp]
    rt.cudaMemcpy.argtypes = [_vp, _vp, _sz, _int]
    rt.cudaGetErrorString.restype = ctypes.c_char_p
    rt.cudaGetErrorString.argtypes = [_int]

    def check(err, what):
        if err != 0:
            raise RuntimeError(f"{what}: {rt.cudaGetErrorString(err).decode()}")

    logits = np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)
    S = T * k
    shapes = {"topk_ids": ((T, k), np.int32), "topk_weights": ((T, k), np.float32),
              "expert_counts": ((E,), np.int32), "expert_offsets": ((E + 1,), np.int32),
              "perm": ((S,), np.int32), "inv_perm": ((S,), np.int32)}
    saved = {"logits": logits}
    for call in range(2):
        check(rt.cudaSetDevice(0), "cudaSetDevice")
        dptr = {}
        for name, nbytes in [("logits", logits.nbytes)] + [
                (n, int(np.prod(s)) * 4) for n, (s, _) in shapes.items()]:
            p = _vp()
            check(rt.cudaMalloc(ctypes.byref(p), nbytes), f"cudaMalloc {name}")
            dptr[name] = p.value
        check(rt.cudaMemcpy(dptr["logits"], logits.ctypes.data, logits.nbytes, H2D), "copy logits")
        st = lib.moe_route_static(dptr["logits"], T, E, k, renorm, dptr["topk_ids"], dptr["topk_weights"],
                                  dptr["expert_counts"], dptr["expert_offsets"], dptr["perm"],
                                  dptr["inv_perm"], None)
        if st != 0:
            raise RuntimeError(f"moe_route_static returned status {st} on call {call}")
        check(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
        for name, (shape, dt) in shapes.items():
            host = np.empty(shape, dtype=dt)
            check(rt.cudaMemcpy(host.ctypes.data, dptr[name], host.nbytes, D2H), f"copy {name}")
            saved[f"{name}{call}"] = host
        if call == 0:
            check(rt.cudaDeviceReset(), "cudaDeviceReset")      # frees every allocation above
        else:
            for p in dptr.values():
                check(rt.cudaFree(p), "cudaFree")
    np.savez(out_path, **saved)


if __name__ == "__main__":
    main()
