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


# Prefill and chunked-prefill workloads (many new tokens per sequence, causal
# among themselves). The first is the chunk of section 7 of "Same GQA,
# Different Execution Cost Across Backends": q_len = 64 new tokens, 32 query
# heads over 8 KV heads, head_dim 64, at the end of a 4096-token context.
PREFILL_CONFIGS = [
    DecodeConfig("chunked_prefill_q64_d64", B=1, sq=64, H=32, G=8, D=64, Tmax=4096, t_lo=4096,
                 t_hi=4096, seed=_BASE_SEED + 21,
                 note="64-token chunk after 4032 cached tokens, 32 heads over 8, D = 64"),
    DecodeConfig("prefill_d64_4k", B=1, sq=4096, H=32, G=8, D=64, Tmax=4096, t_lo=4096,
                 t_hi=4096, seed=_BASE_SEED + 22, note="fresh 4096-token prefill, D = 64"),
    DecodeConfig("prefill_llama3_8b_8k", B=1, sq=8192, H=32, G=8, D=128, Tmax=8192, t_lo=8192,
                 t_hi=8192, seed=_BASE_SEED + 23,
                 note="fresh 8192-token prefill, Llama-3-8B-shaped layer"),
    DecodeConfig("chunked_prefill_llama3_8b", B=4, sq=2048, H=32, G=8, D=128, Tmax=8192,
                 t_lo=8192, t_hi=8192, seed=_BASE_SEED + 24,
                 note="last 2048-token chunk of an 8192-token prompt, 4 sequences"),
]


def config_by_name(name: str) -> DecodeConfig:
    for c in CONFIGS + PREFILL_CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)
