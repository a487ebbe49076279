"""Caches past 2^31 and 2^32 elements: every offset into them must be 64-bit.

The device caches are [B=2, G=8, Tmax=2^21, D=128] bf16 (8 GiB each; the last
unit starts at element 15 * 2^28 > 2^32) and a paged pool whose pages in use
sit above element 2^31. They are allocated with torch.empty: only the valid
rows are written, the rest holds whatever the memory held (NaN included),
which the kernels must never let into a result (decode, fused append, paged
decode, and a prefill chunk on the tcgen05 kernel). The oracle runs on small
host copies (Tmax = 1024) holding the same valid rows -- it reads no entry
past a sequence's length, so its result is the same.
"""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, make_inputs, to_device_bf16

pytestmark = pytest.mark.gpu

B, G, D = 2, 8, 128
TMAX_BIG = 1 << 21
TMAX_SMALL = 1024
LENS = [700, 1000]


def _big_caches(k_small, v_small):
    dk = torch.empty(B, G, TMAX_BIG, D, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(B, G, TMAX_BIG, D, dtype=torch.bfloat16, device="cuda")
    dk[:, :, :TMAX_SMALL].copy_(to_device_bf16(k_small))
    dv[:, :, :TMAX_SMALL].copy_(to_device_bf16(v_small))
    return dk, dv


@pytest.mark.parametrize("H,sq", [(32, 1), (64, 4)], ids=["one-row-tile", "two-row-tiles"])
def test_decode_over_a_cache_past_2_32_elements(H, sq):
    q, k, v, lens = make_inputs(B, sq, H, G, D, TMAX_SMALL, LENS, seed=1201 + H)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    dk, dv = _big_caches(k, v)
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode(to_device_bf16(q), dk, dv, torch.from_numpy(lens).cuda(), scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what=f"big cache H={H}")
    del dk, dv
    torch.cuda.empty_cache()


def test_append_into_a_cache_past_2_32_elements():
    H, sq = 32, 2
    q, k, v, lens = make_inputs(B, sq, H, G, D, TMAX_SMALL, LENS, seed=1301)
    kn = syn.normal_bf16(1302, 1, (B, sq, G, D))
    vn = syn.normal_bf16(1302, 2, (B, sq, G, D))
    scale = 1 / math.sqrt(D)
    k2, v2 = oracle.append_f64(k, v, kn, vn, lens)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k2, v2, lens, scale, threads=8)
    dk, dv = _big_caches(k, v)
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_append(to_device_bf16(q), to_device_bf16(kn), to_device_bf16(vn), dk, dv,
                         torch.from_numpy(lens).cuda(), scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what="append, big cache")
    # The new rows landed at T_b - sq + s of every (b, g), the last of them
    # past element 2^32; the valid rows before them are unchanged.
    got_k = dk[:, :, :TMAX_SMALL].cpu().view(torch.int16).numpy().view(np.uint16)
    got_v = dv[:, :, :TMAX_SMALL].cpu().view(torch.int16).numpy().view(np.uint16)
    for b in range(B):
        T = int(lens[b])
        assert np.array_equal(got_k[b, :, :T], k2[b, :, :T]) and np.array_equal(got_v[b, :, :T], v2[b, :, :T])
    del dk, dv
    torch.cuda.empty_cache()


def test_paged_pool_with_pages_past_2_31_elements():
    """64-token pages in a pool of 2^15 + 64 pages x 8 KV heads x 64 x 128
    elements (4.3 GiB a cache); the sequences' pages are the highest ones."""
    H, sq, ps = 32, 1, 64
    num_pages = (1 << 15) + 64
    q, k, v, lens = make_inputs(B, sq, H, G, D, TMAX_SMALL, LENS, seed=1401)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    max_pages = TMAX_SMALL // ps
    table = np.full((B, max_pages), -1, dtype=np.int32)
    kp = torch.empty(num_pages, G, ps, D, dtype=torch.bfloat16, device="cuda")
    vp = torch.empty(num_pages, G, ps, D, dtype=torch.bfloat16, device="cuda")
    dk_small, dv_small = to_device_bf16(k), to_device_bf16(v)
    nxt = num_pages - 1
    for b in range(B):
        for j in range((int(lens[b]) + ps - 1) // ps):
            table[b, j] = nxt
            kp[nxt].copy_(dk_small[b, :, j * ps:(j + 1) * ps])
            vp[nxt].copy_(dv_small[b, :, j * ps:(j + 1) * ps])
            nxt -= 1
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_paged(to_device_bf16(q), kp, vp, torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                        scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what="paged, big pool")
    del kp, vp
    torch.cuda.empty_cache()


def test_prefill_chunk_over_a_cache_past_2_32_elements():
    """A 64-token chunk (256 rows per KV head: the tcgen05 prefill kernel)
    over the same 2^21-token cache."""
    H, sq = 32, 64
    q, k, v, lens = make_inputs(B, sq, H, G, D, TMAX_SMALL, LENS, seed=1501)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    dk, dv = _big_caches(k, v)
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_prefill(to_device_bf16(q), dk, dv, torch.from_numpy(lens).cuda(), scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what="prefill, big cache")
    del dk, dv
    torch.cuda.empty_cache()
