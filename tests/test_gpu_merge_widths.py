"""Every way the split-KV kernel merges a unit's partials, against the oracle.

The last CTA to arrive on a unit's counter merges the partials of every CTA
that holds part of it (the log-sum-exp rescale of the definition of softmax
over the unit's keys: "GQA analysis", section "Grouped broadcast"). Which code
merges depends on the number of contributors and on the kernel's register
budget: one round of loads for two contributors (four items per thread), for
up to 16 (two items, one row tile at D = 128), for up to 24 or 8 (one item),
and the cooperative three-step merge above that. Here one unit of
contributors x 64 tokens is shared by exactly that many CTAs (the grid forced
with GQA_DECODE_CTAS, one tile each), so each width runs, for each kernel
shape: bf16 with one and two row tiles at D = 128 and 64, and fp8.
"""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, env, make_inputs, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu

WIDTHS = [2, 3, 8, 9, 16, 17, 24, 25, 40]
SHAPES = {                   # (H, G, D, fp8): rows per KV head R = H / G
    "bf16-d128-one-row-tile": (8, 1, 128, False),
    "bf16-d128-two-row-tiles": (32, 1, 128, False),
    "bf16-d64-one-row-tile": (8, 1, 64, False),
    "bf16-d64-two-row-tiles": (32, 1, 64, False),
    "fp8-one-row-tile": (8, 1, 128, True),
    "fp8-two-row-tiles": (32, 1, 128, True),
}


@pytest.mark.parametrize("n", WIDTHS)
@pytest.mark.parametrize("shape", list(SHAPES))
def test_unit_shared_by_n_ctas(shape, n):
    H, G, D, fp8 = SHAPES[shape]
    T = 64 * n - 5                           # a ragged last tile
    q, k, v, lens = make_inputs(1, 1, H, G, D, T, [T], seed=1700 + 37 * n + H + D + fp8)
    scale = 1 / math.sqrt(D)
    plan = gq.gqa_decode_plan(1, 1, H, G, D, T, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["max_tiles"] == n
    with env(GQA_DECODE_CTAS=n):
        if fp8:
            kc, ks = syn.fp8_cache(k, lens)
            vc, vs = syn.fp8_cache(v, lens)
            ref_out, ref_lse = oracle.gqa_decode_fp8_f64(q, kc, vc, ks, vs, lens, scale, threads=8)
            out = torch.empty(1, 1, H, D, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(1, 1, H, dtype=torch.float32, device="cuda")
            gq.gqa_decode_fp8(to_device_bf16(q), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                              torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(),
                              torch.from_numpy(lens).cuda(), scale, out, lse)
            torch.cuda.synchronize()
            assert gq.gqa_decode_check_error() == gq.GQA_OK
            got_out, got_lse = bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)
        else:
            ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
            got_out, got_lse = run_gpu(q, k, v, lens, scale)
    compare(got_out, got_lse, ref_out, ref_lse, what=f"{shape}, {n} contributors")
