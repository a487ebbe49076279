"""The decode variants at the bench's full sizes, in its launch configuration
(default plan): the fp8 cache against the oracle on sampled (sequence, KV head)
units; the paged cache and the fused append bit for bit against the
contiguous path on the same logical cache and the same (m16n8k16) kernel (the
contiguous path is itself checked at these sizes by test_gpu_full_size.py)."""
import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, env, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu

SAMPLE_UNITS = 6


@pytest.mark.parametrize("name", ["llama3_8b_layer", "mqa_end", "long_ctx_b1"])
def test_fp8_full_size_sampled_units(name):
    """Every row of a sampled unit (b, g) -- all (H/G) heads of the group, all
    sq new tokens -- against the oracle over that unit's dequantised cache."""
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg, threads=16)      # NaN past each length
    kc, ks = syn.fp8_cache(k, lens)
    vc, vs = syn.fp8_cache(v, lens)
    del k, v
    out = torch.empty(cfg.B, cfg.sq, cfg.H, cfg.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(cfg.B, cfg.sq, cfg.H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_fp8(to_device_bf16(q), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                      torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(),
                      torch.from_numpy(lens).cuda(), cfg.scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    out, lse = bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)
    hpg = cfg.H // cfg.G
    rng = np.random.default_rng(cfg.seed)
    units = {(0, 0), (cfg.B - 1, cfg.G - 1)}
    while len(units) < min(SAMPLE_UNITS, cfg.B * cfg.G):
        units.add((int(rng.integers(cfg.B)), int(rng.integers(cfg.G))))
    orc = oracle.get()
    for b, g in sorted(units):
        heads = slice(g * hpg, (g + 1) * hpg)
        qs = np.ascontiguousarray(q[b:b + 1, :, heads])
        kd = oracle.dequantize_fp8(kc[b:b + 1, g:g + 1], ks[b:b + 1, g:g + 1])
        vd = oracle.dequantize_fp8(vc[b:b + 1, g:g + 1], vs[b:b + 1, g:g + 1])
        ref_o, ref_l = orc.gqa_decode_kv(qs, kd, vd, lens[b:b + 1], cfg.scale, threads=16)
        compare(out[b:b + 1, :, heads], lse[b:b + 1, :, heads], ref_o, ref_l, what=f"{name} fp8 b={b} g={g}")


@pytest.mark.parametrize("name,page_size", [("llama3_8b_layer", 16), ("llama3_8b_layer", 256), ("mqa_end", 16)])
def test_paged_full_size_equals_contiguous(name, page_size):
    """One row tile (page-major stage at 16-token pages) and two row tiles
    (MQA end: block-major stage). Pages shorter than a tile take every SM
    (no equal-length grid rule), so the contiguous call that must give the
    same bits runs on that grid too (GQA_DECODE_CTAS = the SM count); it is
    also within the parity bar of the contiguous call on its own grid."""
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg, threads=16)
    kp, vp, table = syn.paginate(k, v, lens, page_size, seed=cfg.seed + 100)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with env(GQA_DECODE_CTAS=sms if page_size < 64 else None):
        cont_out, cont_lse = run_gpu(q, k, v, lens, cfg.scale)
    if page_size < 64:
        own_out, own_lse = run_gpu(q, k, v, lens, cfg.scale)
        compare(cont_out, cont_lse, own_out, own_lse, what=f"{name} all-SM grid vs its own")
    out = torch.empty(cfg.B, cfg.sq, cfg.H, cfg.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(cfg.B, cfg.sq, cfg.H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_paged(to_device_bf16(q), to_device_bf16(kp), to_device_bf16(vp),
                        torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), cfg.scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    assert np.array_equal(bf16_to_f64(out), cont_out)
    assert np.array_equal(lse.cpu().numpy().astype(np.float64), cont_lse)


def test_append_full_size_equals_write_then_decode():
    cfg = syn.config_by_name("llama3_8b_layer")
    q, k, v, lens = syn.make_inputs(cfg, threads=16)
    kn = syn.normal_bf16(cfg.seed, 11, (cfg.B, cfg.sq, cfg.G, cfg.D))
    vn = syn.normal_bf16(cfg.seed, 12, (cfg.B, cfg.sq, cfg.G, cfg.D))
    dq, dl = to_device_bf16(q), torch.from_numpy(lens).cuda()
    dk, dv = to_device_bf16(k), to_device_bf16(v)
    out = torch.empty(cfg.B, cfg.sq, cfg.H, cfg.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(cfg.B, cfg.sq, cfg.H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_append(dq, to_device_bf16(kn), to_device_bf16(vn), dk, dv, dl, cfg.scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    k2, v2 = oracle.append_f64(k, v, kn, vn, lens)       # the rows written where the pages say
    assert np.array_equal(dk.cpu().view(torch.int16).numpy().view(np.uint16), k2)
    assert np.array_equal(dv.cpu().view(torch.int16).numpy().view(np.uint16), v2)
    ref_out, ref_lse = run_gpu(q, k2, v2, lens, cfg.scale)
    assert np.array_equal(bf16_to_f64(out), ref_out)
    assert np.array_equal(lse.cpu().numpy().astype(np.float64), ref_lse)
