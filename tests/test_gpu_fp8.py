"""fp8 (E4M3, one scale per 64-token block) cache decode on the GPU against the
oracle over the dequantised cache, within the parity bar."""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, make_inputs, min_tiles, to_device_bf16

pytestmark = pytest.mark.gpu


def _run_fp8(q, kc, vc, ks, vs, lens, scale):
    B, sq, H, D = q.shape
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_fp8(to_device_bf16(q), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                      torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(),
                      torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda(), scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("split", [1, None], ids=["split1", "default"])
@pytest.mark.parametrize("H,G,sq", [(32, 8, 1), (8, 8, 1), (32, 1, 1), (64, 8, 4), (12, 4, 3)], ids=str)
def test_fp8_matches_oracle(H, G, sq, split):
    lens = [1, 15, 63, 64, 65, 200, 300, 0]
    B, D, Tmax = len(lens), 128, 300
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=800 + H + G + sq)
    kc, ks = syn.fp8_cache(k, lens)
    vc, vs = syn.fp8_cache(v, lens)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_fp8_f64(q, kc, vc, ks, vs, lens, scale, threads=8)
    with min_tiles(split):
        out, lse = _run_fp8(q, kc, vc, ks, vs, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"fp8 H={H} G={G} sq={sq}")


def test_fp8_scales_act_per_block():
    """Scaling one block's codes' scale by 2 changes the result exactly as the
    oracle says (the kernel applies each 64-token block's own scale)."""
    B, sq, H, G, D, Tmax = 2, 1, 16, 2, 128, 256
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [256, 190], seed=820)
    kc, ks = syn.fp8_cache(k, lens)
    vc, vs = syn.fp8_cache(v, lens)
    ks[0, 1, 2] *= 2.0
    vs[1, 0, 1] *= 0.5
    ref_out, ref_lse = oracle.gqa_decode_fp8_f64(q, kc, vc, ks, vs, lens, 0.09)
    out, lse = _run_fp8(q, kc, vc, ks, vs, lens, 0.09)
    compare(out, lse, ref_out, ref_lse, what="fp8 per-block scales")


@pytest.mark.parametrize("H,G", [(32, 8), (64, 2)], ids=["one-row-tile", "two-row-tiles"])
def test_fp8_zero_block_scales(H, G):
    """A block scale of 0 (an all-zero block, as a caller may store it): a
    zero K scale makes that block's scores exactly 0, a zero V scale its
    values 0, including in the first block of a unit and on a unit's every
    block."""
    B, sq, D, Tmax = 3, 1, 128, 256
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [256, 200, 130], seed=822 + H)
    kc, ks = syn.fp8_cache(k, lens)
    vc, vs = syn.fp8_cache(v, lens)
    last = G - 1
    ks[0, 0, 0] = 0.0          # first block of a unit
    vs[0, 0, 0] = 0.0
    vs[1, last, 2] = 0.0       # a later block
    ks[1, 0, 1] = 0.0
    vs[2, last, :] = 0.0       # every block of a unit: out = 0 there
    ref_out, ref_lse = oracle.gqa_decode_fp8_f64(q, kc, vc, ks, vs, lens, 0.09)
    with min_tiles(1):
        out, lse = _run_fp8(q, kc, vc, ks, vs, lens, 0.09)
    compare(out, lse, ref_out, ref_lse, what=f"fp8 zero block scales H={H} G={G}")
    hpg = H // G
    assert np.all(out[2, :, last * hpg:(last + 1) * hpg] == 0.0)


def test_fp8_rejects_head_dim_64():
    q, k, v, lens = make_inputs(1, 1, 8, 2, 64, 64, [64], seed=821)
    kc = torch.zeros(1, 2, 64, 64, dtype=torch.uint8, device="cuda")
    sc = torch.ones(1, 2, 1, dtype=torch.float32, device="cuda")
    out = torch.empty(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gq.GQADecodeError) as e:
        gq.gqa_decode_fp8(to_device_bf16(q), kc, kc, sc, sc, torch.from_numpy(lens).cuda(), 0.1, out)
    assert e.value.status == gq.GQA_ERR_UNSUPPORTED
