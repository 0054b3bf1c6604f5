"""The synthetic workloads the path is checked and measured on.

Each stands in for a workload the pages describe (text at n=4096 with 12
heads, Long-Range-Arena-length batches, the BigBird block layout, a long
sequence); the public suites themselves are not used.  All draw Q, K, V from
``synthetic.qkv`` and the graph from seed 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dtype: str                    # "fp32" | "bf16"
    kind: str                     # "token" | "causal" (token graph cut to j <= i) | "block"
    r: int = 0                    # token graph: window radius
    n_globals: int = 0            # token graph: globals at positions 0..g-1
    rand_per_row: int = 0         # token graph: random draws per row
    block: int = 0                # block graph: tokens per block
    window_blocks: int = 0
    rand_blocks: int = 0
    global_blocks: int = 0
    hops: int = 5
    alpha: float = 0.1
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def units(self) -> int:
        return self.B * self.H

    def graph_args(self) -> dict:
        if self.kind in ("token", "causal"):
            return dict(n=self.n, r=self.r, n_globals=self.n_globals,
                        rand_per_row=self.rand_per_row, seed=self.seed)
        return dict(n=self.n, block=self.block, window_blocks=self.window_blocks,
                    rand_blocks=self.rand_blocks, global_blocks=self.global_blocks,
                    seed=self.seed)

    def describe(self) -> dict:
        d = dict(workload=self.name, batch=self.B, heads=self.H, seq_len=self.n, d_head=self.d,
                 io_dtype=self.dtype, graph=self.kind, hops=self.hops, alpha=self.alpha)
        d.update({k: v for k, v in self.graph_args().items() if k != "n"})
        return d


TINY = Workload("tiny_fp32_n512", 1, 1, 512, 64, "fp32", "token", r=32, n_globals=4,
                rand_per_row=8)
TEXT = Workload("text_bf16_b2h12_n4096", 2, 12, 4096, 64, "bf16", "token", r=256,
                n_globals=16, rand_per_row=32)
LRA = Workload("lra_bf16_b32h8_n1024", 32, 8, 1024, 64, "bf16", "token", r=32, n_globals=8,
               rand_per_row=16)
BIGBIRD = Workload("bigbird_itc_bf16_b4h12_n4096", 4, 12, 4096, 64, "bf16", "block", block=64,
                   window_blocks=3, rand_blocks=3, global_blocks=2)
LONG = Workload("long_bf16_b1h16_n16384", 1, 16, 16384, 64, "bf16", "token", r=256,
                n_globals=32, rand_per_row=32)

ALL = (TINY, TEXT, LRA, BIGBIRD, LONG)

# The causal variant of the text workload: the same sizes on the lower-triangular
# graph that autoregressive use needs (Diffuser notes sec 2.6).
CAUSAL_TEXT = Workload("causal_text_bf16_b2h12_n4096", 2, 12, 4096, 64, "bf16", "causal", r=256,
                       n_globals=16, rand_per_row=32)
# The text workload's pattern (r 256, 16 globals, 32 draws per row) over a length sweep
# (n = 4096 is TEXT itself).
SWEEP = tuple(Workload(f"text_bf16_b2h12_n{n}", 2, 12, n, 64, "bf16", "token", r=256,
                       n_globals=16, rand_per_row=32) for n in (1024, 2048, 8192, 16384))
VARIANTS = (CAUSAL_TEXT,) + SWEEP
BY_NAME = {w.name: w for w in ALL + VARIANTS}
