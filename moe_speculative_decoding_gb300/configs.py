"""The workloads: synthetic MoE layers shaped like the models the pages measure.

Each entry fixes shapes, dtypes, the pass sizes n and the routing-reuse values rho of
one workload.  Shapes follow the public model cards of the named models; the pages use
the same models ("Speculative Decoding for Mixture-of-Experts Models" (Lan), §2 "Setup"
and §4.4).  No arithmetic of the method lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    index: int                 # stream id used by synth.seed_for
    name: str
    d: int                     # hidden size
    f: int                     # expert intermediate size
    N: int                     # routed experts
    m: int                     # experts per token
    w_dtype: str               # "bf16" or "f32"
    x_dtype: str
    n_values: tuple            # pass sizes
    rhos: tuple                # routing reuse of the synthetic traces
    layers: int = 1
    n_shared: int = 0          # always-on shared experts (gate 1)
    f_shared: int = 0
    windows: int = 64          # passes per n (non-overlapping windows of the trace)
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def expert_bytes(self) -> int:
        return 3 * self.d * self.f * (2 if self.w_dtype == "bf16" else 4)


TINY = Workload(0, "tiny-fp32", d=256, f=512, N=8, m=2, w_dtype="f32", x_dtype="f32",
                n_values=(4,), rhos=(0.0,), windows=1,
                notes="router W_r[8,256] ~ N(0,1/d); logits = x W_r^T; seed 0")
DSV2_LITE = Workload(1, "deepseek-v2-lite-layer", d=2048, f=1408, N=64, m=6, w_dtype="bf16",
                     x_dtype="bf16", n_values=tuple(range(1, 9)), rhos=(0.0, 0.3, 0.6),
                     n_shared=2, f_shared=1408)
QWEN3 = Workload(2, "qwen3-30b-a3b-layer", d=2048, f=768, N=128, m=8, w_dtype="bf16",
                 x_dtype="bf16", n_values=tuple(range(1, 17)), rhos=(0.0, 0.5))
MIXTRAL = Workload(3, "mixtral-8x7b-layer", d=4096, f=14336, N=8, m=2, w_dtype="bf16",
                   x_dtype="bf16", n_values=tuple(range(1, 9)), rhos=(0.0, 0.8))
QWEN3_STACK = Workload(4, "qwen3-30b-a3b-48-layer-expert-stack", d=2048, f=768, N=128, m=8,
                       w_dtype="bf16", x_dtype="bf16", n_values=tuple(range(1, 17)),
                       rhos=(0.4,), layers=48, windows=16,
                       notes="48 layers resident (57.98 GB bf16); one shared pass x for all layers")

WORKLOADS = (TINY, DSV2_LITE, QWEN3, MIXTRAL, QWEN3_STACK)
BY_NAME = {w.name: w for w in WORKLOADS}
