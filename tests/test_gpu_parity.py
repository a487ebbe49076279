"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small cases run the oracle on every row: they span several 64-token tiles,
ragged tails, empty and short sequences, both head dimensions, the MHA and
MQA ends, sq = 4 causal rows, and plans that split units across many CTAs.
"""
import math

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
import synthetic as syn
from gpu_helpers import bf16_to_f64, compare, make_inputs, min_tiles, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu

HEAD_SHAPES = [  # (H, G, sq): R = (H/G)*sq rows per KV head
    (32, 8, 1),   # GQA group 4
    (8, 8, 1),    # MHA end
    (32, 1, 1),   # MQA end, R = 32
    (16, 2, 2),   # R = 16
    (64, 8, 4),   # ragged-workload heads, R = 32
    (8, 1, 4),    # MQA with 4 new tokens, R = 32
    (12, 4, 3),   # R = 9, odd sizes
]
LENS = [1, 15, 16, 17, 63, 64, 65, 200]


@pytest.mark.parametrize("min_tiles_per_cta", [1, None], ids=["split1", "default"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,G,sq", HEAD_SHAPES, ids=lambda x: str(x))
def test_sweep_vs_oracle(H, G, sq, D, min_tiles_per_cta):
    B, Tmax = len(LENS), 256
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, LENS, seed=100 + H + G + sq + D)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    with min_tiles(min_tiles_per_cta):
        out, lse = run_gpu(q, k, v, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"H={H} G={G} sq={sq} D={D}")


def test_tiny_workload_all_rows():
    cfg = syn.config_by_name("tiny_gqa_d64")
    q, k, v, lens = syn.make_inputs(cfg)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, cfg.scale, threads=8)
    for mt in (1, None):
        with min_tiles(mt):
            out, lse = run_gpu(q, k, v, lens, cfg.scale)
        compare(out, lse, ref_out, ref_lse, what=cfg.name)


def test_empty_and_short_sequences():
    """T_b = 0 (no key at all) and T_b < sq (the first rows see nothing): those
    rows are out = 0, lse = -inf; the rest match the oracle."""
    lens = [0, 1, 2, 3, 4, 5, 0, 70]
    q, k, v, lens = make_inputs(len(lens), 4, 16, 4, 128, 96, lens, seed=200)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.09, threads=8)
    for mt in (1, None):
        with min_tiles(mt):
            out, lse = run_gpu(q, k, v, lens, 0.09)
        compare(out, lse, ref_out, ref_lse, what="short")


def test_all_sequences_empty():
    q, k, v, lens = make_inputs(3, 1, 8, 2, 64, 64, [0, 0, 0], seed=201)
    out, lse = run_gpu(q, k, v, lens, 0.125)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_lengths_past_tmax_are_clamped():
    Tmax = 80
    q, k, v, _ = make_inputs(2, 1, 8, 2, 128, Tmax, [Tmax, Tmax], seed=202)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, np.array([Tmax, Tmax], np.int32), 0.1)
    out, lse = run_gpu(q, k, v, np.array([Tmax + 1000, 2 ** 30], np.int32), 0.1)
    compare(out, lse, ref_out, ref_lse, what="clamp")
    # negative lengths read as 0
    out, lse = run_gpu(q, k, v, np.array([-5, Tmax], np.int32), 0.1)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


def test_tmax_not_a_multiple_of_the_tile():
    """The last tile of each unit runs past Tmax; those rows come from the
    tensor map's out-of-bounds fill, not from the next unit's memory."""
    Tmax = 100
    q, k, v, lens = make_inputs(3, 2, 16, 4, 64, Tmax, [100, 99, 37], seed=203)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.2)
    for mt in (1, None):
        with min_tiles(mt):
            out, lse = run_gpu(q, k, v, lens, 0.2)
        compare(out, lse, ref_out, ref_lse, what="Tmax%64")


def test_head_mapping_table_on_gpu(request):
    """The printed Exaone4 table (32 query heads over 8 KV heads): with V of KV
    head g constant g+1, out[h] must be kv(h)+1 (neighbouring KV heads differ
    by 1, far outside the 1e-2 bar)."""
    from oracle_pins import load_mapping_table
    table = load_mapping_table()
    H, G, D, T = 32, 8, 64, 333
    q = syn.normal_bf16(300, 1, (1, 1, H, D))
    k = syn.normal_bf16(300, 2, (1, G, T, D))
    v = np.empty((1, G, T, D), dtype=np.uint16)
    for g in range(G):
        v[0, g] = syn.f32_to_bf16_bits(np.float32(g + 1))
    for mt in (1, None):
        with min_tiles(mt):
            out, _ = run_gpu(q, k, v, np.array([T], np.int32), 0.125)
        for h in range(H):
            np.testing.assert_allclose(out[0, 0, h], table[h] + 1.0, atol=1e-2, rtol=0)


def test_dominant_key_anywhere():
    """A key that beats the others by a wide margin returns its V row, whichever
    tile, slice or CTA share it falls in."""
    D, T = 128, 700
    for tstar in (0, 63, 64, 333, 699):
        q = np.full((1, 1, 4, D), syn.f32_to_bf16_bits(np.float32(1.0))[0], dtype=np.uint16)
        k = syn.normal_bf16(301, 2, (1, 1, T, D))
        v = syn.normal_bf16(301, 3, (1, 1, T, D))
        k[0, 0, tstar] = syn.f32_to_bf16_bits(np.float32(4.0))[0]
        with min_tiles(1):
            out, lse = run_gpu(q, k, v, np.array([T], np.int32), 1 / math.sqrt(D))
        ref = syn.bf16_bits_to_f32(v[0, 0, tstar]).astype(np.float64)
        for h in range(4):
            np.testing.assert_allclose(out[0, 0, h], ref, atol=1e-2 * max(1, np.abs(ref).max()), rtol=0)


def test_no_lse_pointer():
    q, k, v, lens = make_inputs(2, 1, 32, 8, 128, 128, [128, 50], seed=204)
    ref_out, _ = oracle.gqa_decode_f64(q, k, v, lens, 0.1)
    out, _ = run_gpu(q, k, v, lens, 0.1, with_lse=False)
    assert np.abs(out - ref_out).max() <= 1e-2


def test_explicit_workspace_matches_library_workspace():
    q, k, v, lens = make_inputs(4, 2, 16, 2, 128, 512, [512, 300, 1, 64], seed=205)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out1 = torch.empty(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    lse1 = torch.empty(4, 2, 16, dtype=torch.float32, device="cuda")
    out2, lse2 = torch.empty_like(out1), torch.empty_like(lse1)
    with min_tiles(1):
        gq.gqa_decode(dq, dk, dv, dl, 0.1, out1, lse1)
        nbytes = gq.gqa_decode_workspace_bytes(4, 2, 16, 2, 128, 512)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        gq.gqa_decode_ex(dq, dk, dv, dl, 0.1, out2, lse2, ws)
        with pytest.raises(gq.GQADecodeError) as e:
            gq.gqa_decode_ex(dq, dk, dv, dl, 0.1, out2, lse2, ws[: nbytes - 256])
        assert e.value.status == gq.GQA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_explicit_workspace_guard_words():
    """Canary bytes on both sides of a caller-owned workspace stay untouched by
    a call whose plan splits units over many CTAs (every CTA writes partial
    slots, the counters are used), and the result matches the oracle. The
    workspace starts as those canary bytes too: it needs no clearing."""
    B, sq, H, G, D, Tmax = 3, 4, 64, 8, 128, 900
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [900, 517, 77], seed=208)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    guard = 4096
    with min_tiles(1):
        nbytes = gq.gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax)
        buf = torch.full((nbytes + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
        ws = buf[guard:guard + nbytes]
        assert ws.data_ptr() % 256 == 0
        for _ in range(2):
            gq.gqa_decode_ex(dq, dk, dv, dl, 1 / math.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    host = buf.cpu().numpy()
    assert np.all(host[:guard] == 0xA5) and np.all(host[guard + nbytes:] == 0xA5), "workspace guard"
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 1 / math.sqrt(D), threads=8)
    compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what="guarded workspace")


def test_prefill_partials_leave_the_decode_counters_alone():
    """A short prefill chunk whose key ranges are split writes its partials
    into a library buffer of its own, not over the decode workspace's arrival
    counters: a split-KV decode on the same stream right after it matches the
    oracle with a clean status word, and so does the prefill."""
    B, sq, H, G, D, Tmax = 1, 64, 8, 2, 128, 2048
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [2048], seed=212)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    out, lse = run_gpu(q, k, v, lens, scale, entry=gq.gqa_prefill)
    compare(out, lse, ref_out, ref_lse, what="split prefill")
    q2, k2, v2, lens2 = make_inputs(3, 1, 32, 8, 128, 700, [700, 650, 129], seed=213)
    ref2 = oracle.gqa_decode_f64(q2, k2, v2, lens2, scale, threads=8)
    with min_tiles(1):
        out2, lse2 = run_gpu(q2, k2, v2, lens2, scale)   # checks the status word
    compare(out2, lse2, *ref2, what="decode after split prefill")


def test_release_workspace_frees_and_the_next_call_allocates_again():
    """gqa_decode_release_workspace gives the (device, stream) buffer back:
    the device's free memory grows by about its size, and the next call on
    the stream allocates a new one and is still correct."""
    B, sq, H, G, D, Tmax = 64, 1, 32, 1, 128, 2048
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [2048] * B, seed=209)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out = torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, sq, H, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    need = gq.gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax)
    assert need > 2 << 20
    gq.gqa_decode(dq, dk, dv, dl, 1 / math.sqrt(D), out, lse, stream=s)
    s.synchronize()
    free_held, _ = torch.cuda.mem_get_info()
    gq.gqa_decode_release_workspace(s)
    free_released, _ = torch.cuda.mem_get_info()
    assert free_released - free_held >= need // 2, (free_held, free_released, need)
    gq.gqa_decode_release_workspace(s)          # nothing held: still fine
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 1 / math.sqrt(D), threads=8)
    gq.gqa_decode(dq, dk, dv, dl, 1 / math.sqrt(D), out, lse, stream=s)
    s.synchronize()
    assert gq.gqa_decode_check_error(s) == gq.GQA_OK
    compare(bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse, what="after release")
    gq.gqa_decode_release_workspace(s)


def test_repeated_calls_are_bit_identical():
    q, k, v, lens = make_inputs(3, 1, 64, 8, 128, 1000, [1000, 999, 640], seed=206)
    a, la = run_gpu(q, k, v, lens, 0.09)
    b, lb = run_gpu(q, k, v, lens, 0.09)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_argument_errors_on_gpu():
    q, k, v, lens = make_inputs(1, 1, 8, 2, 128, 64, [64], seed=207)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out = torch.empty(1, 1, 8, 128, dtype=torch.bfloat16, device="cuda")
    # misaligned output pointer (a view two elements into a buffer)
    buf = torch.empty(8 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    bad = buf[2:2 + 8 * 128].view(1, 1, 8, 128)
    with pytest.raises(gq.GQADecodeError) as e:
        gq.gqa_decode(dq, dk, dv, dl, 0.1, bad, None)
    assert e.value.status == gq.GQA_ERR_MISALIGNED
    with pytest.raises(TypeError):
        gq.gqa_decode(dq.float(), dk, dv, dl, 0.1, out, None)
    assert gq.gqa_decode_check_error() == gq.GQA_OK


@pytest.mark.parametrize("H,G,sq", [(4, 2, 1), (6, 2, 1), (10, 2, 1), (6, 1, 1), (7, 1, 1),
                                    (24, 1, 1), (31, 1, 1), (5, 1, 5), (3, 1, 9)],
                         ids=lambda x: str(x))
def test_every_row_count(H, G, sq):
    """Row counts R = (H/G)*sq that are not multiples of anything: partial
    slots, padded MMA rows and the combine's addressing for each."""
    lens = [1, 70, 129, 300]
    B, Tmax, D = len(lens), 320, 128
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=400 + H * 7 + G + sq)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.1, threads=8)
    for mt in (1, 3):
        with min_tiles(mt):
            out, lse = run_gpu(q, k, v, lens, 0.1)
        compare(out, lse, ref_out, ref_lse, what=f"R={H // G * sq}")


@pytest.mark.parametrize("B,sq,H,G,D,lens", [
    (2, 8, 32, 4, 128, [700, 9]),     # speculative-style: 8 new tokens, group of 8, R = 64
    (3, 2, 48, 2, 64, [300, 1, 0]),   # R = 48, a sequence shorter than sq, an empty one
], ids=["R64", "R48"])
def test_decode_with_more_than_32_rows_per_kv_head(B, sq, H, G, D, lens):
    """gqa_decode takes any number of rows per KV head; above 32 it runs the
    prefill kernel on the same definition."""
    q, k, v, lens = make_inputs(B, sq, H, G, D, 700, lens, seed=210 + H)
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    out, lse = run_gpu(q, k, v, lens, scale)
    compare(out, lse, ref_out, ref_lse, what=f"decode R={(H // G) * sq}")


@pytest.mark.parametrize("sq,H,G,ragged", [(1, 8, 2, True), (4, 16, 2, True), (1, 8, 2, False)],
                         ids=["one-row-tile", "two-row-tiles", "equal-lengths"])
def test_more_than_256_sequences(sq, H, G, ragged):
    """300 sequences: the work partition keeps the first 256 lengths in
    registers and reads the rest again; shares must start and end at the
    right sequence past that point too. Equal lengths take the rule that
    shrinks the grid to a whole number of units per CTA (600 units)."""
    B, D, Tmax = 300, 64, 96
    if ragged:
        lens = syn.uniform_int(5150 + sq, syn.STREAM_LENS, B, 0, Tmax)
    else:
        lens = np.full(B, 64, dtype=np.int32)
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, lens, seed=5160 + sq + int(ragged))
    scale = 1 / math.sqrt(D)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    for mt in (1, None):
        with min_tiles(mt):
            out, lse = run_gpu(q, k, v, lens, scale)
        compare(out, lse, ref_out, ref_lse, what=f"B=300 sq={sq} ragged={ragged} min_tiles={mt}")
