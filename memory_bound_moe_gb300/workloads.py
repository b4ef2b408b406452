"""Seeded synthetic workloads for the MoE glue path.

This module only draws random numbers; it holds none of the method's
arithmetic. Both the CUDA path (through the tests and the benchmark) and the
CPU oracle receive the very same host bytes produced here.

Shapes follow the MoE deployments the pages discuss (a Qwen3-30B-A3B-like
layer with intermediate size 768 in "[FlashInfer] CUTLASS MoE kernel
optimisation", section 2 "Dynamic threads"; prefill versus decode in "CuTeDSL
at Perplexity", section "Prefill and decode specialization"; the odd token
count 1023 used as a non-power-of-two edge case in the vLLM fused indexer-Q
analysis, test section). No public dataset or model weights are involved.

Recipe (seed 0 unless stated): one CPU ``torch.Generator`` draws, in this
order, the router logits ``[T, E]`` (float32 standard normal, plus a
per-expert bias), the token activations ``x [T, H]``, the fc1 output
``gate_up [T*k, 2I]`` and the fc2 output ``expert_out [T*k, H]`` (float32
normal with standard deviation ``act_std``, rounded to bfloat16).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    H: int          # hidden size
    E: int          # experts
    k: int          # experts per token
    renorm: bool    # renormalise the k selected softmax weights
    I: int          # expert intermediate size (gate_up has 2I columns)
    act_std: float = 1.0
    hot_experts: tuple = field(default=())   # experts that get +hot_bias
    hot_bias: float = 0.0
    note: str = ""

    @property
    def S(self) -> int:
        """Number of (token, expert) slots, T*k."""
        return self.T * self.k

    def describe(self) -> str:
        return (f"{self.name}: T={self.T} H={self.H} E={self.E} top-{self.k}"
                f"{' renorm' if self.renorm else ' softmax'} I={self.I}")


WORKLOADS = {
    "tiny": Workload("tiny", T=64, H=256, E=8, k=2, renorm=True, I=128,
                     note="small case the oracle finishes instantly"),
    "mid": Workload("mid", T=4096, H=2048, E=128, k=8, renorm=True, I=768,
                    note="Qwen3-30B-A3B-like layer; the throughput workload"),
    "decode": Workload("decode", T=16, H=7168, E=256, k=8, renorm=False, I=2048,
                       note="decode regime: latency per call"),
    "prefill": Workload("prefill", T=8192, H=4096, E=8, k=2, renorm=True, I=14336,
                        note="prefill regime: few experts, wide intermediate"),
    "skewed": Workload("skewed", T=1023, H=2880, E=32, k=4, renorm=True, I=2880,
                       act_std=2.0, hot_experts=(0, 1, 2, 3), hot_bias=3.0,
                       note="odd sizes; experts 0-3 take most tokens"),
}


def custom(name: str, T: int, H: int, E: int, k: int, renorm: bool, I: int,
           act_std: float = 1.0, hot_experts=(), hot_bias: float = 0.0) -> Workload:
    return Workload(name, T, H, E, k, renorm, I, act_std, tuple(hot_experts), hot_bias)


def generate(w: Workload, seed: int = 0, parts=("logits", "x", "gate_up", "expert_out")):
    """Draw the workload's inputs on the CPU. Parts are always drawn in the
    fixed order logits, x, gate_up, expert_out from one generator; parts not
    requested are still drawn (so the others keep their values) unless they
    come after every requested part."""
    order = ("logits", "x", "gate_up", "expert_out")
    want = set(parts)
    last = max(order.index(p) for p in want)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {}
    for idx, part in enumerate(order[: last + 1]):
        if part == "logits":
            t = torch.randn((w.T, w.E), generator=g, dtype=torch.float32)
            if w.hot_experts:
                t[:, list(w.hot_experts)] += w.hot_bias
        elif part == "x":
            t = (torch.randn((w.T, w.H), generator=g, dtype=torch.float32) * w.act_std).to(torch.bfloat16)
        elif part == "gate_up":
            t = (torch.randn((w.S, 2 * w.I), generator=g, dtype=torch.float32) * w.act_std).to(torch.bfloat16)
        else:
            t = (torch.randn((w.S, w.H), generator=g, dtype=torch.float32) * w.act_std).to(torch.bfloat16)
        if part in want:
            out[part] = t
    return out


def as_u16(t: torch.Tensor):
    """A CPU bfloat16 tensor's bit patterns as a numpy uint16 array (no copy of values)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_u16(a) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU bfloat16 tensor."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
