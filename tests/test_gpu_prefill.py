"""Prefill / chunked-prefill kernel (gqa_prefill, tcgen05) vs the fp64 oracle.

The oracle is the decode definition itself -- new token s of sequence b at
position T_b - sq + s sees keys t <= T_b - sq + s of KV head h / (H/G) -- which
holds for any number of new tokens. Cases span several 128-row and 128-token
tiles with ragged tails, fresh prefills (T_b = sq) and chunks behind earlier
context, head groups of 1 (MHA) to 32 (MQA) including non-powers of two, both
head dimensions, lengths shorter than sq (rows that see nothing), empty
sequences, Tmax not a multiple of the tile, and NaN in every cache entry past
a sequence's length.
"""
import contextlib
import math
import os

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import compare, make_inputs, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu


def prefill(*args, **kw):
    return run_gpu(*args, entry=gq.gqa_prefill, **kw)


@contextlib.contextmanager
def forced_splits(n):
    """Key ranges per pair of row tiles (None: the library's plan)."""
    old = os.environ.get("GQA_PREFILL_SPLITS")
    if n is None:
        os.environ.pop("GQA_PREFILL_SPLITS", None)
    else:
        os.environ["GQA_PREFILL_SPLITS"] = str(n)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("GQA_PREFILL_SPLITS", None)
        else:
            os.environ["GQA_PREFILL_SPLITS"] = old


CASES = [  # (B, sq, H, G, D, Tmax, lens)
    (1, 64, 32, 8, 64, 4096, [4096]),          # the page's chunk: 64 new tokens after 4032
    (2, 300, 8, 2, 128, 300, [300, 300]),      # fresh prefill, ragged last row tile
    (3, 50, 12, 4, 64, 450, [50, 177, 400]),   # group of 3, chunks behind context
    (2, 130, 4, 4, 128, 260, [130, 259]),      # MHA end (group 1)
    (1, 40, 32, 1, 128, 200, [200]),           # MQA end: 1280 rows over one KV head
    (2, 257, 2, 1, 64, 700, [257, 690]),       # group 2, odd sizes
    (4, 8, 16, 4, 128, 129, [8, 3, 0, 129]),   # T_b < sq and T_b = 0
]


@pytest.mark.parametrize("B,sq,H,G,D,Tmax,lens", CASES, ids=lambda x: str(x))
def test_prefill_vs_oracle(B, sq, H, G, D, Tmax, lens):
    """Each case in the library's plan, and with every pair's key range split
    over 3 and over 7 CTAs (partials merged by the combine kernel; ranges that
    hold no visible key for some rows, and more ranges than key tiles)."""
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=700 + B + sq + H + G + D)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=16)
    for n in (None, 3, 7):
        with forced_splits(n):
            out, lse = prefill(q, k, v, lens, scale)
        compare(out, lse, ref_out, ref_lse, what=f"prefill B={B} sq={sq} H={H} G={G} D={D} splits={n}")


def test_prefill_equals_decode_definition_small_rows():
    """Where both entry points apply (R <= 32) they compute the same thing."""
    q, k, v, lens = make_inputs(3, 4, 16, 2, 128, 1000, [1000, 517, 4], seed=731)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.09, threads=16)
    a, la = run_gpu(q, k, v, lens, 0.09)
    b, lb = prefill(q, k, v, lens, 0.09)
    compare(a, la, ref_out, ref_lse, what="decode")
    compare(b, lb, ref_out, ref_lse, what="prefill")


def test_prefill_sharp_softmax_and_rescale():
    """Scores that grow along the sequence force the running max up tile after
    tile (the O rescale path); one dominant key per row is an O(1) output."""
    B, sq, H, G, D, T = 1, 256, 4, 1, 128, 640
    q, k, v, lens = make_inputs(B, sq, H, G, D, T, [T], seed=732)
    kf = syn.bf16_bits_to_f32(k).astype(np.float32)
    ramp = np.linspace(0.2, 3.0, T, dtype=np.float32)[None, None, :, None]
    k = syn.f32_to_bf16_bits((kf * ramp).astype(np.float32))
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.3, threads=16)
    out, lse = prefill(q, k, v, lens, 0.3)
    compare(out, lse, ref_out, ref_lse, what="ramp")


def test_prefill_repeated_calls_are_bit_identical():
    q, k, v, lens = make_inputs(2, 200, 8, 2, 64, 900, [900, 333], seed=733)
    a, la = prefill(q, k, v, lens, 0.125)
    b, lb = prefill(q, k, v, lens, 0.125)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_prefill_no_lse_pointer():
    q, k, v, lens = make_inputs(1, 128, 8, 2, 128, 300, [300], seed=734)
    ref_out, _ = oracle.gqa_decode_f64(q, k, v, lens, 0.1, threads=16)
    out, _ = prefill(q, k, v, lens, 0.1, with_lse=False)
    assert np.abs(out - ref_out).max() <= 1e-2


def test_prefill_argument_errors_on_gpu():
    q, k, v, lens = make_inputs(1, 16, 8, 2, 128, 64, [64], seed=735)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    buf = torch.empty(16 * 8 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    bad = buf[2:2 + 16 * 8 * 128].view(1, 16, 8, 128)
    with pytest.raises(gq.GQADecodeError) as e:
        gq.gqa_prefill(dq, dk, dv, dl, 0.1, bad, None)
    assert e.value.status == gq.GQA_ERR_MISALIGNED


@pytest.mark.parametrize("name", [c.name for c in syn.PREFILL_CONFIGS])
def test_prefill_workloads_sampled(name):
    """The bench's prefill workloads at full size, in the bench's launch
    configuration: sampled new tokens (every head) against the oracle. Token s
    of a prefill is the single-token call at length T_b - sq + s + 1 on the
    same cache (the causal-prefix pin of the oracle)."""
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg, threads=16)
    out, lse = prefill(q, k, v, lens, cfg.scale)
    rng = np.random.default_rng(cfg.seed)
    picks = sorted(set([0, cfg.sq - 1, min(127, cfg.sq - 1), min(128, cfg.sq - 1)] +
                       list(rng.integers(0, cfg.sq, 4))))
    for b in range(cfg.B):
        for s in picks:
            t = int(lens[b]) - cfg.sq + s + 1
            qs = np.ascontiguousarray(q[b:b + 1, s:s + 1])
            ref_o, ref_l = oracle.gqa_decode_f64(qs, k[b:b + 1], v[b:b + 1],
                                                 np.array([t], np.int32), cfg.scale, threads=16)
            compare(out[b:b + 1, s:s + 1], lse[b:b + 1, s:s + 1], ref_o, ref_l, what=f"{name} b={b} s={s}")
