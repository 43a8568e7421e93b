"""The five WKV7 workloads the library is checked and measured on.

Each is named by what it is. ``storage`` is the dtype of r, w, k, v, a, b,
dy and y; the state, checkpoints and gradients are always float32.
``s_init_std`` None means a zero initial state. ``ckpt_every`` is the forward
checkpoint interval the backward consumes.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    N: int
    storage: str
    s_init_std: float | None
    ckpt_every: int

    @property
    def width(self) -> int:
        """Model width H*N (called C in RWKV-7's own notation)."""
        return self.H * self.N

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny-fp32", 1, 64, 2, 16, "f32", None, 16),
        Workload("small-fp32-carry", 2, 512, 4, 64, "f32", 0.1, 16),
        Workload("rwkv7-0.1b-layer-fp32", 8, 4096, 12, 64, "f32", None, 16),
        Workload("rwkv7-1.5b-layer-bf16", 4, 4096, 32, 64, "bf16", None, 16),
        Workload("long-carry-fp32", 1, 65536, 40, 64, "f32", 0.1, 16),
    )
}

# The throughput workload: the RWKV-7 1.5B-shaped layer scan.
BENCH_WORKLOAD = "rwkv7-1.5b-layer-bf16"
