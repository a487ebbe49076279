"""Failure detection on the GPU without a fault: every device-side wait of the
kernel is bounded. With the test hook GQA_DECODE_DEBUG_SKIP_TILE, CTA 0 never
loads one of its K/V tiles, so its consumers' wait for it expires (after the
200 ms GQA_DECODE_DEBUG_TIMEOUT_MS); the kernel records that in the status
word, waits for its own copies in flight and returns. The host must read
GQA_ERR_DEVICE_TIMEOUT, and the context must stay usable: the next call,
without the hook, is correct."""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
from gpu_helpers import compare, make_inputs, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,G,sq", [(32, 8, 1), (64, 8, 4)], ids=["one-row-tile", "two-row-tiles"])
def test_expired_wait_is_reported_and_the_context_survives(monkeypatch, H, G, sq):
    B, D, Tmax = 2, 128, 700
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [700, 650], seed=77 + H)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    assert gq.gqa_decode_check_error() == gq.GQA_OK

    monkeypatch.setenv("GQA_DECODE_DEBUG_TIMEOUT_MS", "200")
    monkeypatch.setenv("GQA_DECODE_DEBUG_SKIP_TILE", "1")
    gq.gqa_decode(dq, dk, dv, dl, 1 / math.sqrt(D), out, lse)
    assert gq.gqa_decode_check_error() == gq.GQA_ERR_DEVICE_TIMEOUT
    assert gq.gqa_decode_check_error() == gq.GQA_OK   # reading clears the word

    monkeypatch.delenv("GQA_DECODE_DEBUG_SKIP_TILE")
    monkeypatch.delenv("GQA_DECODE_DEBUG_TIMEOUT_MS")
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 1 / math.sqrt(D), threads=8)
    for _ in range(2):   # every SM's tensor memory is allocatable again
        got_out, got_lse = run_gpu(q, k, v, lens, 1 / math.sqrt(D), device_inputs=(dq, dk, dv, dl))
        compare(got_out, got_lse, ref_out, ref_lse, what="after timeout")


def test_prefill_expired_wait_is_reported_and_the_context_survives(monkeypatch):
    """The tcgen05 prefill kernel on the same hook: CTA 0's MMA warps wait for a
    K tile that never comes, give up, let the products they issued finish, and
    the CTA frees its tensor memory before returning (a later launch on that SM
    allocates it again). The next call, without the hook, matches the oracle."""
    B, sq, H, G, D, Tmax = 1, 300, 8, 2, 128, 700
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [700], seed=91)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    assert gq.gqa_decode_check_error() == gq.GQA_OK

    monkeypatch.setenv("GQA_DECODE_DEBUG_TIMEOUT_MS", "200")
    monkeypatch.setenv("GQA_DECODE_DEBUG_SKIP_TILE", "1")
    gq.gqa_prefill(dq, dk, dv, dl, 1 / math.sqrt(D), out, lse)
    assert gq.gqa_decode_check_error() == gq.GQA_ERR_DEVICE_TIMEOUT
    assert gq.gqa_decode_check_error() == gq.GQA_OK

    monkeypatch.delenv("GQA_DECODE_DEBUG_SKIP_TILE")
    monkeypatch.delenv("GQA_DECODE_DEBUG_TIMEOUT_MS")
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 1 / math.sqrt(D), threads=8)
    for _ in range(2):   # every SM's tensor memory is allocatable again
        got_out, got_lse = run_gpu(q, k, v, lens, 1 / math.sqrt(D), device_inputs=(dq, dk, dv, dl),
                                   entry=gq.gqa_prefill)
        compare(got_out, got_lse, ref_out, ref_lse, what="prefill after timeout")


@pytest.mark.parametrize("H,G,sq", [(32, 8, 1), (64, 8, 4)], ids=["one-row-tile", "two-row-tiles"])
def test_timed_out_call_leaves_the_counters_clean(monkeypatch, H, G, sq):
    """A call whose wait expires must still leave every unit's arrival counter
    at zero. A CUDA-graph replay carries the counter tag (epoch) of the call
    that was captured; a count left part-way by a timed-out replay would let
    the next replay merge a unit before all its partials are written, with
    the status word clean. Here every call carries the same tag
    (GQA_DECODE_DEBUG_EPOCH), as graph replays do. With 2 x 8 units of 11
    tiles over 11 CTAs, CTA 0's share is unit 0 whole and the first 5 tiles
    of unit 1; it gives up in unit 0, before it counts its arrival on unit 1.
    The next calls get new values, so a merge that read a stale partial
    would not match the oracle."""
    B, D, Tmax = 2, 128, 700
    scale = 1 / math.sqrt(D)
    monkeypatch.setenv("GQA_DECODE_DEBUG_EPOCH", "4242")
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [700, 650], seed=301 + H)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    plan = gq.gqa_decode_plan(B, sq, H, G, D, Tmax, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["ctas"] == 11, plan   # the share the docstring works out

    monkeypatch.setenv("GQA_DECODE_DEBUG_TIMEOUT_MS", "200")
    monkeypatch.setenv("GQA_DECODE_DEBUG_SKIP_TILE", "1")
    gq.gqa_decode(dq, dk, dv, dl, scale, out, lse)
    assert gq.gqa_decode_check_error() == gq.GQA_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("GQA_DECODE_DEBUG_SKIP_TILE")
    monkeypatch.delenv("GQA_DECODE_DEBUG_TIMEOUT_MS")

    for rep in range(2):
        q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [700, 650], seed=302 + H + rep)
        dq.copy_(to_device_bf16(q)); dk.copy_(to_device_bf16(k)); dv.copy_(to_device_bf16(v))
        ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
        got_out, got_lse = run_gpu(q, k, v, lens, scale, device_inputs=(dq, dk, dv, dl))
        compare(got_out, got_lse, ref_out, ref_lse, what=f"same tag after a timeout, call {rep}")
