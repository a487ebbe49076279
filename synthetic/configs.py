"""The decode workloads, named by what they are, with their sizes.

Every workload draws Q, K and V i.i.d. N(0,1) rounded to bf16 from its own seed;
the scale is 1/sqrt(D). Per-sequence lengths T_b count the valid cache entries
including the sq new tokens (the new tokens' K/V are appended before attending,
as in the incremental decode loop of "GQA analysis", section "Incremental
decode"). Ragged lengths are uniform integers in [t_lo, t_hi], both inclusive.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    sq: int
    H: int
    G: int
    D: int
    Tmax: int
    t_lo: int
    t_hi: int
    seed: int
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def group(self) -> int:
        return self.H // self.G

    @property
    def rows(self) -> int:
        """R = (H/G)*sq query rows share one KV head."""
        return self.group * self.sq

    def asdict(self):
        return {k: getattr(self, k) for k in
                ("name", "B", "sq", "H", "G", "D", "Tmax", "t_lo", "t_hi", "seed")}


_BASE_SEED = 20261202

CONFIGS = [
    DecodeConfig("tiny_gqa_d64", B=1, sq=1, H=32, G=8, D=64, Tmax=1024, t_lo=1024, t_hi=1024,
                 seed=_BASE_SEED + 1,
                 note="Exaone4-1.2B-like head layout (32 query heads over 8 KV heads)"),
    DecodeConfig("llama3_8b_layer", B=16, sq=1, H=32, G=8, D=128, Tmax=4096, t_lo=4096,
                 t_hi=4096, seed=_BASE_SEED + 2, note="Llama-3-8B-shaped layer"),
    DecodeConfig("mha_end", B=8, sq=1, H=32, G=32, D=128, Tmax=4096, t_lo=4096, t_hi=4096,
                 seed=_BASE_SEED + 3, note="G = H"),
    DecodeConfig("mqa_end", B=64, sq=1, H=32, G=1, D=128, Tmax=8192, t_lo=8192, t_hi=8192,
                 seed=_BASE_SEED + 4, note="G = 1"),
    DecodeConfig("long_ctx_b1", B=1, sq=1, H=64, G=8, D=128, Tmax=131072, t_lo=131072,
                 t_hi=131072, seed=_BASE_SEED + 5, note="long context, batch 1"),
    DecodeConfig("long_ctx_b4", B=4, sq=1, H=64, G=8, D=128, Tmax=131072, t_lo=131072,
                 t_hi=131072, seed=_BASE_SEED + 6, note="long context, batch 4"),
    DecodeConfig("ragged_sq4", B=64, sq=4, H=64, G=8, D=128, Tmax=32768, t_lo=512,
                 t_hi=32768, seed=_BASE_SEED + 7,
                 note="speculative-style: 4 new tokens, causal among them, ragged lengths"),
]


def config_by_name(name: str) -> DecodeConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)
