"""The opt-in tcgen05 decode kernel (GQA_DECODE_TC=1; 17..32 rows per KV head,
bf16, D = 128) against the fp64 oracle, element by element, through the C ABI
-- and the default m16n8k16 split-KV kernel on the same inputs.

Lengths straddle the 128-token tiles of the tensor-core kernel (and the
64-token ones of the other): empty, shorter than sq, one key, 127/128/129,
several tiles with a ragged tail. Plans: the default, one tile per CTA (units
split over many CTAs; more CTAs than tiles), and forced grids of 3 and 37
CTAs (segments that start and end inside units, so merges of 2..many
contributors and CTAs that carry two partials).
"""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_helpers import compare, env, make_inputs, min_tiles, run_gpu

pytestmark = pytest.mark.gpu

SHAPES = [  # (H, G, sq) with R = (H/G)*sq in 17..32
    (32, 1, 1),   # MQA end, R = 32
    (64, 8, 4),   # ragged-workload heads, R = 32 (causal among 4 new tokens)
    (24, 1, 1),   # R = 24: rows 24..31 of the MMA's N unused
    (8, 2, 5),    # R = 20, sq = 5
    (17, 1, 1),   # R = 17
]
LENS = [0, 3, 1, 127, 128, 129, 300, 513, 1000]


PLANS = [("default", None, None), ("split1", 1, None), ("ctas3", None, 3), ("ctas37", None, 37)]


@pytest.mark.parametrize("tc", ["1", "0"], ids=["tcgen05", "mma_sync"])
@pytest.mark.parametrize("plan", PLANS, ids=[p[0] for p in PLANS])
@pytest.mark.parametrize("H,G,sq", SHAPES, ids=str)
def test_two_row_tile_shapes_vs_oracle(H, G, sq, plan, tc):
    D, Tmax = 128, 1024
    B = len(LENS)
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, LENS, seed=300 + H + G + sq)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    _, mt, ctas = plan
    with min_tiles(mt), env(GQA_DECODE_TC=tc, GQA_DECODE_CTAS=ctas):
        out, lse = run_gpu(q, k, v, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"H={H} G={G} sq={sq} plan={plan[0]} tc={tc}")


def test_large_scores_move_the_max_late():
    """Scores that grow along the sequence: each later tile raises some rows'
    max by more than the rescale slack, so O^T is rescaled in tensor memory
    many times within a segment (and across split segments)."""
    B, sq, H, G, D, Tmax = 2, 1, 32, 1, 128, 1024
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [1024, 900], seed=411)
    # K rows scaled up with position (bf16-exact powers of two): later keys
    # dominate, with gaps far above 2^8 in the exponent.
    ramp = (2.0 ** np.floor(np.arange(Tmax) / 128.0)).astype(np.float32)[None, None, :, None]
    k = syn.f32_to_bf16_bits(syn.bf16_bits_to_f32(k) * ramp)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    for ctas in (None, 5):
        with env(GQA_DECODE_CTAS=ctas, GQA_DECODE_TC="1"):
            out, lse = run_gpu(q, k, v, lens, scale)
        compare(out, lse, ref_out, ref_lse, what=f"growing scores ctas={ctas}")


@pytest.mark.parametrize("name", ["mqa_end", "ragged_sq4"])
def test_full_size_sampled_units_both_kernels(name):
    """The bench workloads at full size, default plan: sampled (sequence, KV
    head) units against the oracle, for the tcgen05 and m16n8k16 kernels."""
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg, threads=16)
    hpg = cfg.H // cfg.G
    rng = np.random.default_rng(cfg.seed + 7)
    units = {(0, 0), (cfg.B - 1, cfg.G - 1)}
    while len(units) < 5:
        units.add((int(rng.integers(cfg.B)), int(rng.integers(cfg.G))))
    orc = oracle.get()
    refs = {}
    for b, g in sorted(units):
        heads = slice(g * hpg, (g + 1) * hpg)
        refs[(b, g)] = orc.gqa_decode(np.ascontiguousarray(q[b:b + 1, :, heads]),
                                         np.ascontiguousarray(k[b:b + 1, g:g + 1]),
                                         np.ascontiguousarray(v[b:b + 1, g:g + 1]), lens[b:b + 1], cfg.scale,
                                         threads=16)
    for tc in ("1", "0"):
        with env(GQA_DECODE_TC=tc):
            out, lse = run_gpu(q, k, v, lens, cfg.scale)
        for (b, g), (ro, rl) in refs.items():
            heads = slice(g * hpg, (g + 1) * hpg)
            compare(out[b:b + 1, :, heads], lse[b:b + 1, :, heads], ro, rl, what=f"{name} tc={tc} b={b} g={g}")
