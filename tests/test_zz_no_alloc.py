"""gqa_decode_noalloc, the entry point for callers that must not allocate
device memory while running (a serving engine that gave all device memory to
its own pool at start-up, a plugin handed tensors but no allocator, a loop
that cannot take cudaMalloc's implicit synchronisation).

Its output, called through the C ABI twice in a row, must match the regular
gqa_decode entry point's within the parity tolerance; problems too large for
its fixed scratch array must be refused before anything is enqueued. Kept in a
file of its own that pytest collects last, and written to pass both alone in a
fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
from gpu_helpers import compare, make_inputs, min_tiles, to_device_bf16

pytestmark = pytest.mark.gpu


def _abi_noalloc(dq, dk, dv, dl, scale, out, lse):
    B, sq, H, D = dq.shape
    _, G, Tmax, _ = dk.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return gq.load().gqa_decode_noalloc(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                        dl.data_ptr(), scale, out.data_ptr(), lse.data_ptr(),
                                        B, sq, H, G, D, Tmax, stream)


@pytest.mark.parametrize("shape", [(6, 1, 32, 8, 128, 700), (3, 4, 64, 8, 128, 400),
                                   (2, 1, 32, 1, 64, 900)], ids=str)
@pytest.mark.parametrize("split", [1, None], ids=["many-splits", "default"])
def test_noalloc_matches_regular_entry_point(shape, split):
    B, sq, H, G, D, Tmax = shape
    lens = np.linspace(sq, Tmax, B).astype(np.int32)
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=900 + B + H)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    scale = D ** -0.5
    with min_tiles(split):
        ref = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
        gq.gqa_decode(dq, dk, dv, dl, scale, ref, ref_lse)
        for _ in range(2):  # the scratch keeps the previous call's contents
            out = torch.full_like(ref, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            assert _abi_noalloc(dq, dk, dv, dl, scale, out, lse) == gq.GQA_OK
            torch.cuda.synchronize()
            assert gq.gqa_decode_check_error() == gq.GQA_OK
            compare(out.float().cpu().numpy().astype(np.float64),
                    lse.cpu().numpy().astype(np.float64),
                    ref.float().cpu().numpy().astype(np.float64),
                    ref_lse.cpu().numpy().astype(np.float64), what="noalloc")


def test_noalloc_refuses_problems_beyond_its_scratch():
    # 2^21 one-token sequences need 32 MiB of arrival counters alone (8 B per
    # sequence, KV head and row tile), more than the fixed array holds; the
    # call must be refused up front.
    B = 1 << 21
    need = gq.gqa_decode_workspace_bytes(B, 1, 1, 1, 64, 64)
    assert need > gq.GQA_NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    rc = gq.load().gqa_decode_noalloc(p, p, p, lens.data_ptr(), 0.125, p, None,
                                      B, 1, 1, 1, 64, 64, None)
    assert rc == gq.GQA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK


def test_noalloc_refuses_more_than_32_rows_per_kv_head():
    # gqa_decode sends (H/G)*sq > 32 rows to the prefill kernel, whose split
    # key ranges use a library-allocated workspace; the allocation-free entry
    # point does not, and refuses such shapes before anything is enqueued.
    B, sq, H, G, D, Tmax = 1, 1, 64, 1, 128, 256
    dq = torch.zeros(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    dk = torch.zeros(B, G, Tmax, D, dtype=torch.bfloat16, device="cuda")
    dl = torch.full((B,), Tmax, dtype=torch.int32, device="cuda")
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    assert _abi_noalloc(dq, dk, dk, dl, D ** -0.5, out, lse) == gq.GQA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
