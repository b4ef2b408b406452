"""QK RMSNorm (in place) on the GPU through the C ABI, against the oracle.
bfloat16 output of float32 arithmetic: |gpu - ref| <= 2e-2 + 1e-2 |ref|."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import check_bf16_close

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


@pytest.mark.parametrize("T,nq,nk,hd", [(1, 32, 4, 128), (7, 8, 8, 64), (4096, 32, 4, 128),
                                        (333, 16, 2, 256), (50, 0, 4, 128), (50, 4, 0, 64),
                                        (8192, 64, 8, 128)])
@pytest.mark.parametrize("bias", [0.0, 1.0])
def test_qk_rmsnorm_matches_oracle(dev, oracle_mod, T, nq, nk, hd, bias):
    from memory_bound_moe_gb300 import moe_qk_rmsnorm
    O = oracle_mod
    rng = np.random.default_rng(T + nq + hd)
    q = O.bf16_round(rng.standard_normal((T, nq, hd)) * np.exp(rng.uniform(-4, 4, (T, nq, 1))))
    k = O.bf16_round(rng.standard_normal((T, nk, hd)) * 3)
    qw = O.bf16_round(rng.standard_normal(hd) * 0.2)
    kw = O.bf16_round(rng.standard_normal(hd) * 0.2)
    eps = 1e-6
    qd, kd = bf16_dev(q, dev), bf16_dev(k, dev)
    moe_qk_rmsnorm(qd, kd, bf16_dev(qw, dev), bf16_dev(kw, dev), bias, eps)
    torch.cuda.synchronize()
    rq, rk = O.qk_norm(q, k, qw, kw, bias, eps)
    if nq:
        check_bf16_close(u16(qd), rq, f"q T={T} nq={nq} hd={hd}")
    if nk:
        check_bf16_close(u16(kd), rk, f"k T={T} nk={nk} hd={hd}")


def test_qk_rmsnorm_zero_heads_and_eps(dev, oracle_mod):
    from memory_bound_moe_gb300 import moe_qk_rmsnorm
    O = oracle_mod
    hd = 128
    q = np.zeros((4, 2, hd), dtype=np.uint16)            # all-zero heads: 0 * rsqrt(eps) = 0
    q[1, 1] = O.bf16_round(np.full(hd, 2.0))
    k = O.bf16_round(np.tile([1.0, -1.0], hd // 2)[None, None, :].repeat(4, 0))
    w = O.bf16_round(np.zeros(hd))
    qd, kd = bf16_dev(q, dev), bf16_dev(k, dev)
    moe_qk_rmsnorm(qd, kd, bf16_dev(w, dev), bf16_dev(w, dev), 1.0, 3.0)
    torch.cuda.synchronize()
    check_bf16_close(u16(qd), O.qk_norm(q, k, w, w, 1.0, 3.0)[0], "zero heads")
    assert np.all(O.bf16_decode(u16(kd)) == np.tile([0.5, -0.5], hd // 2))   # 1/sqrt(1+3)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_qk_rmsnorm_16_byte_aligned_buffers(dev, oracle_mod, hd):
    """q, k and the weights 16 but not 32 bytes aligned: the 16-byte-vector
    shape of the kernel, against the oracle."""
    from memory_bound_moe_gb300 import moe_qk_rmsnorm
    O = oracle_mod
    rng = np.random.default_rng(hd)
    T, nq, nk = 37, 6, 2
    q = O.bf16_round(rng.standard_normal((T, nq, hd)))
    k = O.bf16_round(rng.standard_normal((T, nk, hd)) * 2)
    qw = O.bf16_round(rng.standard_normal(hd) * 0.5)
    kw = O.bf16_round(rng.standard_normal(hd) * 0.5)

    def shifted(a):   # a device copy that starts 16 bytes past a 256-byte boundary
        flat = bf16_dev(a.reshape(-1), dev)
        buf = torch.empty(flat.numel() + 8, dtype=torch.bfloat16, device=dev)
        view = buf[8:8 + flat.numel()]
        view.copy_(flat)
        assert view.data_ptr() % 32 == 16
        return buf, view.view(a.shape)

    _, qd = shifted(q)
    _, kd = shifted(k)
    _, qwd = shifted(qw)
    _, kwd = shifted(kw)
    moe_qk_rmsnorm(qd, kd, qwd, kwd, 0.0, 1e-6)
    torch.cuda.synchronize()
    rq, rk = O.qk_norm(q, k, qw, kw, 0.0, 1e-6)
    check_bf16_close(u16(qd), rq, f"q hd={hd} (16-byte aligned)")
    check_bf16_close(u16(kd), rk, f"k hd={hd} (16-byte aligned)")
