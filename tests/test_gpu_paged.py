"""Paged-cache decode on the GPU: against the oracle over the logical cache,
and bit for bit against the contiguous path on the same logical cache."""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, make_inputs, min_tiles, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu


def _run_paged(q, kp, vp, table, lens, scale):
    B, sq, H, D = q.shape
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_paged(to_device_bf16(q), to_device_bf16(kp), to_device_bf16(vp),
                        torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("split", [1, None], ids=["split1", "default"])
@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,G,sq", [(32, 8, 1), (64, 8, 4), (8, 1, 4)], ids=str)
def test_paged_matches_oracle_and_contiguous(H, G, sq, D, page_size, split):
    lens = [1, 15, 64, 65, 200, 511, 512, 0]
    B, Tmax = len(lens), 512
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=700 + H + sq + D + page_size)
    kp, vp, table = syn.paginate(k, v, lens, page_size, seed=701 + page_size)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_paged_f64(q, kp, vp, table, lens, scale, threads=8)
    with min_tiles(split):
        out, lse = _run_paged(q, kp, vp, table, lens, scale)
        cont_out, cont_lse = run_gpu(q, k, v, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"paged ps={page_size}")
    assert np.array_equal(out, cont_out) and np.array_equal(lse, cont_lse)


def test_paged_rejects_bad_page_sizes():
    q, k, v, lens = make_inputs(1, 1, 8, 2, 64, 64, [64], seed=710)
    kp, vp, table = syn.paginate(k, v, lens, 16, seed=711)
    dq, dkp, dvp = to_device_bf16(q), to_device_bf16(kp), to_device_bf16(vp)
    out = torch.empty(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    dl, dt = torch.from_numpy(lens).cuda(), torch.from_numpy(table).cuda()
    lib = gq.load()
    for ps, code in ((12, gq.GQA_ERR_UNSUPPORTED), (8, gq.GQA_ERR_UNSUPPORTED), (0, gq.GQA_ERR_INVALID_ARG)):
        rc = lib.gqa_decode_paged(dq.data_ptr(), dkp.data_ptr(), dvp.data_ptr(), dt.data_ptr(),
                                  dl.data_ptr(), 0.1, out.data_ptr(), None, 1, 1, 8, 2, 64, ps,
                                  kp.shape[0], table.shape[1], None)
        assert rc == code, ps


@pytest.mark.parametrize("page_size", [16, 64])
def test_out_of_range_page_reads_as_zeros(page_size):
    """A block-table entry outside [0, num_pages) for a page the sequence uses
    reads as zeros (no fault): the result is the oracle's over the logical
    cache with that page's rows zero. 16-token pages go through the producer's
    lane copies, 64-token pages through TMA boxes."""
    lens = [200, 130]
    B, sq, H, G, D, Tmax = 2, 1, 16, 4, 128, 256
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=720 + page_size)
    kp, vp, table = syn.paginate(k, v, lens, page_size, seed=721)
    bad_b, bad_j = 0, 1                      # second page of sequence 0
    table = table.copy()
    table[bad_b, bad_j] = kp.shape[0] + 3
    k0, v0 = k.copy(), v.copy()
    rows = slice(bad_j * page_size, (bad_j + 1) * page_size)
    k0[bad_b, :, rows, :] = 0
    v0[bad_b, :, rows, :] = 0
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k0, v0, lens, scale, threads=8)
    out, lse = _run_paged(q, kp, vp, table, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"bad page ps={page_size}")
