"""CUDA-graph capture and replay, the way a serving loop runs decode steps.

One call on the capture stream sizes the library's workspace; the next call
is captured into a torch.cuda.CUDAGraph and replayed with new contents of the
same input tensors (values and sequence lengths). Every replay must match the
oracle. The plans split units over many CTAs, so each replay goes through
partial slots, the per-unit arrival counters and the last-arriver merge --
with the epoch of the captured call, which the counters must not remember
from one replay to the next.
"""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, env, make_inputs, min_tiles, to_device_bf16

pytestmark = pytest.mark.gpu

REPLAYS = 3


def _graph(fn, stream):
    with torch.cuda.stream(stream):
        fn()                       # sizes the workspace of this stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def _lens(rng, B, Tmax, sq):
    return rng.integers(sq, Tmax + 1, size=B).astype(np.int32)


@pytest.mark.parametrize("H,G,sq", [(32, 8, 1), (64, 8, 4), (32, 1, 1)],
                         ids=["one-row-tile", "two-row-tiles", "mqa-two-row-tiles"])
def test_decode_graph_replays(H, G, sq):
    B, D, Tmax = 3, 128, 1500
    rng = np.random.default_rng(1701 + H + sq)
    scale = 1 / math.sqrt(D)
    dq = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(B, G, Tmax, D, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    dl = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")

    def load(seed):
        q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, _lens(rng, B, Tmax, sq), seed=seed)
        dq.copy_(to_device_bf16(q)); dk.copy_(to_device_bf16(k)); dv.copy_(to_device_bf16(v))
        dl.copy_(torch.from_numpy(lens))
        return q, k, v, lens

    load(1800)
    s = torch.cuda.Stream()
    with min_tiles(1):
        g = _graph(lambda: gq.gqa_decode(dq, dk, dv, dl, scale, out, lse), s)
    for rep in range(REPLAYS):
        q, k, v, lens = load(1801 + rep)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert gq.gqa_decode_check_error() == gq.GQA_OK
        ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
        compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
                what=f"graph replay {rep} H={H} sq={sq}")


def test_variant_graph_replays():
    """fp8, paged and fused-append steps captured together in one graph."""
    B, sq, H, G, D, Tmax, ps = 3, 2, 32, 8, 128, 1024, 16
    rng = np.random.default_rng(1901)
    scale = 1 / math.sqrt(D)
    dq = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    dl = torch.empty(B, dtype=torch.int32, device="cuda")
    # fp8
    k8 = torch.empty(B, G, Tmax, D, dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty(B, G, Tmax // 64, dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    # paged (every page of every sequence, so the table can stay fixed)
    num_pages = B * (Tmax // ps) + 3
    kp = torch.empty(num_pages, G, ps, D, dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    tab = torch.empty(B, Tmax // ps, dtype=torch.int32, device="cuda")
    # append
    kc = torch.empty(B, G, Tmax, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    kn = torch.empty(B, sq, G, D, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    outs = [torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    lses = [torch.empty(B, sq, H, dtype=torch.float32, device="cuda") for _ in range(3)]

    def load(seed):
        lens = _lens(rng, B, Tmax, sq)
        q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=seed)
        dq.copy_(to_device_bf16(q)); dl.copy_(torch.from_numpy(lens))
        kcode, kscale = syn.fp8_cache(k, lens)
        vcode, vscale = syn.fp8_cache(v, lens)
        k8.copy_(torch.from_numpy(kcode)); v8.copy_(torch.from_numpy(vcode))
        ks.copy_(torch.from_numpy(kscale).reshape(ks.shape)); vs.copy_(torch.from_numpy(vscale).reshape(vs.shape))
        kpn, vpn, table = syn.paginate(k, v, np.full(B, Tmax, np.int32), ps, seed=seed, spare_pages=3)
        kp.copy_(to_device_bf16(kpn)); vp.copy_(to_device_bf16(vpn)); tab.copy_(torch.from_numpy(table))
        knew = syn.normal_bf16(seed, 11, (B, sq, G, D))
        vnew = syn.normal_bf16(seed, 12, (B, sq, G, D))
        kc.copy_(to_device_bf16(k)); vc.copy_(to_device_bf16(v))
        kn.copy_(to_device_bf16(knew)); vn.copy_(to_device_bf16(vnew))
        return q, k, v, lens, (kcode, kscale, vcode, vscale), knew, vnew

    load(2000)

    def step():
        gq.gqa_decode_fp8(dq, k8, v8, ks, vs, dl, scale, outs[0], lses[0])
        gq.gqa_decode_paged(dq, kp, vp, tab, dl, scale, outs[1], lses[1])
        gq.gqa_decode_append(dq, kn, vn, kc, vc, dl, scale, outs[2], lses[2])

    s = torch.cuda.Stream()
    with min_tiles(1):
        g = _graph(step, s)
    for rep in range(REPLAYS):
        q, k, v, lens, f8, knew, vnew = load(2001 + rep)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert gq.gqa_decode_check_error() == gq.GQA_OK
        got = [(bf16_to_f64(o), l.cpu().numpy().astype(np.float64)) for o, l in zip(outs, lses)]
        kd, vd = oracle.dequantize_fp8(f8[0], f8[1]), oracle.dequantize_fp8(f8[2], f8[3])
        ro, rl = oracle.get().gqa_decode_kv(q, kd, vd, lens, scale, threads=8)
        compare(*got[0], ro, rl, what=f"graph replay {rep} fp8")
        ro, rl = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
        compare(*got[1], ro, rl, what=f"graph replay {rep} paged")
        k2, v2 = oracle.append_f64(k, v, knew, vnew, lens)
        ro, rl = oracle.gqa_decode_f64(q, k2, v2, lens, scale, threads=8)
        compare(*got[2], ro, rl, what=f"graph replay {rep} append")


def test_prefill_graph_replays():
    """A 64-token chunk with its key range split over CTAs (partials and the
    combine kernel), captured and replayed with new lengths."""
    B, sq, H, G, D, Tmax = 2, 64, 32, 8, 128, 2048
    rng = np.random.default_rng(2101)
    scale = 1 / math.sqrt(D)
    dq = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(B, G, Tmax, D, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    dl = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")

    def load(seed):
        q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, _lens(rng, B, Tmax, sq), seed=seed)
        dq.copy_(to_device_bf16(q)); dk.copy_(to_device_bf16(k)); dv.copy_(to_device_bf16(v))
        dl.copy_(torch.from_numpy(lens))
        return q, k, v, lens

    load(2200)
    s = torch.cuda.Stream()
    with env(GQA_PREFILL_SPLITS=5):
        g = _graph(lambda: gq.gqa_prefill(dq, dk, dv, dl, scale, out, lse), s)
    for rep in range(REPLAYS):
        q, k, v, lens = load(2201 + rep)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert gq.gqa_decode_check_error() == gq.GQA_OK
        ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
        compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
                what=f"graph replay {rep} prefill")


def test_noalloc_entry_graph_replays():
    """The allocation-free entry (a fixed per-device scratch array) captured and
    replayed like the others."""
    B, sq, H, G, D, Tmax = 3, 2, 32, 8, 128, 1500
    rng = np.random.default_rng(2501)
    scale = 1 / math.sqrt(D)
    dq = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(B, G, Tmax, D, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    dl = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")

    def load(seed):
        q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, _lens(rng, B, Tmax, sq), seed=seed)
        dq.copy_(to_device_bf16(q)); dk.copy_(to_device_bf16(k)); dv.copy_(to_device_bf16(v))
        dl.copy_(torch.from_numpy(lens))
        return q, k, v, lens

    load(2600)
    s = torch.cuda.Stream()
    with min_tiles(1):
        g = _graph(lambda: gq.gqa_decode_noalloc(dq, dk, dv, dl, scale, out, lse), s)
    for rep in range(REPLAYS):
        q, k, v, lens = load(2601 + rep)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert gq.gqa_decode_check_error() == gq.GQA_OK
        ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
        compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
                what=f"graph replay {rep} noalloc")


def test_chained_steps_read_the_previous_steps_output():
    """Each step's output is the next step's Q. The decode kernel is launched
    with programmatic dependent launch, so its prologue may overlap the step
    before it; it must read no input before that step has finished writing."""
    B, sq, H, G, D, Tmax = 2, 1, 32, 8, 128, 1800
    scale = 1 / math.sqrt(D)
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [1800, 950], seed=2701)
    dk, dv, dl = to_device_bf16(k), to_device_bf16(v), torch.from_numpy(lens).cuda()
    bufs = [to_device_bf16(q)] + [torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    with min_tiles(1):
        for i in range(4):
            gq.gqa_decode(bufs[i], dk, dv, dl, scale, bufs[i + 1], lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    # Step 4 against the oracle on step 3's actual output (its bf16 bits).
    q3 = bufs[3].cpu().view(torch.int16).numpy().view(np.uint16)
    ref_out, ref_lse = oracle.gqa_decode_f64(q3, k, v, lens, scale, threads=8)
    compare(bf16_to_f64(bufs[4]), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what="chained step 4")
