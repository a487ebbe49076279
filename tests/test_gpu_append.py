"""Fused append + decode on the GPU against the oracle: the output and LSE
within the parity bar, the updated caches bit for bit (the new rows at
T_b - sq + s, every other entry, NaN tails included, unchanged)."""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, make_inputs, min_tiles, to_device_bf16

pytestmark = pytest.mark.gpu


def _run_append(q, k, v, kn, vn, lens, scale):
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dkn, dvn = to_device_bf16(kn), to_device_bf16(vn)
    dl = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    B, sq, H, D = q.shape
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_append(dq, dkn, dvn, dk, dv, dl, scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    kc = dk.view(torch.int16).cpu().numpy().view(np.uint16)
    vc = dv.view(torch.int16).cpu().numpy().view(np.uint16)
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), kc, vc


@pytest.mark.parametrize("split", [1, None], ids=["split1", "default"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,G,sq", [(32, 8, 1), (16, 2, 2), (64, 8, 4), (8, 1, 4)], ids=str)
def test_append_matches_oracle(H, G, sq, D, split):
    # lengths that put the new rows at the start, across 64-token tile
    # boundaries, at Tmax, and partly below position 0
    lens = [1, 2, 64, 65, 66, 130, 300, 3]
    B, Tmax = len(lens), 300
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=600 + H + G + sq + D)
    kn = syn.normal_bf16(601 + D, 1, (B, sq, G, D))
    vn = syn.normal_bf16(601 + D, 2, (B, sq, G, D))
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse, ref_k, ref_v = oracle.gqa_decode_append_f64(q, k, v, kn, vn, lens, scale,
                                                                  threads=8)
    with min_tiles(split):
        out, lse, kc, vc = _run_append(q, k, v, kn, vn, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"append H={H} G={G} sq={sq} D={D}")
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


def test_append_equals_write_then_decode():
    """The fused call and 'write the rows, then gqa_decode' give the same bits."""
    B, sq, H, G, D, Tmax = 4, 2, 32, 8, 128, 500
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [500, 129, 64, 7], seed=610)
    kn = syn.normal_bf16(611, 1, (B, sq, G, D))
    vn = syn.normal_bf16(611, 2, (B, sq, G, D))
    out, lse, kc, vc = _run_append(q, k, v, kn, vn, lens, 0.09)
    k2, v2 = oracle.append_f64(k, v, kn, vn, lens)
    dk2, dv2 = to_device_bf16(k2), to_device_bf16(v2)
    dq, dl = to_device_bf16(q), torch.from_numpy(lens).cuda()
    out2 = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse2 = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode(dq, dk2, dv2, dl, 0.09, out2, lse2)
    torch.cuda.synchronize()
    assert np.array_equal(out, bf16_to_f64(out2))
    assert np.array_equal(lse, lse2.cpu().numpy().astype(np.float64))
