"""The fp8 cache on the CPU: the oracle's E4M3 decoding against PyTorch's
float8_e4m3fn, the double-valued oracle against the pinned bf16 one, and the
generator's codes and scales."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from oracle_pins import _f64, make_case


def test_e4m3_decoding_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_double_valued_oracle_equals_the_bf16_oracle():
    """Fed the same values, the two entry points give the same bits: the one
    for double K/V is tied to the pinned bf16 one."""
    for (B, sq, H, G, D, Tmax, lens) in [(2, 1, 8, 2, 16, 30, [30, 7]), (1, 4, 8, 1, 8, 20, [20])]:
        q, k, v, lens = make_case(B, sq, H, G, D, Tmax, lens, seed=80)
        a_out, a_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.3)
        b_out, b_lse = oracle.get().gqa_decode_kv(q, _f64(k), _f64(v), lens, 0.3)
        assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)


def test_generator_codes_and_scales():
    lens = np.array([130, 64, 0], dtype=np.int32)
    k = syn.fill_cache(3, 2, 3, 2, 200, 128, lens, syn.BF16_NAN)
    codes, scales = syn.fp8_cache(k, lens)
    assert codes.shape == k.shape and scales.shape == (3, 2, 4)
    deq = oracle.dequantize_fp8(codes, scales)
    for b, T in enumerate(lens):
        x = _f64(k[b, :, :T])
        if T:
            # block amax maps to at most 448; quantisation error within half an e4m3 step
            assert np.all(np.abs(deq[b, :, :T] - x) <= 2.0 ** -4 * np.abs(x) + 2.0 ** -9 * scales.max())
        assert np.all(codes[b, :, T:] == syn.E4M3_NAN)
    assert np.all(scales[2] == 1.0)


def _block_scale_pin_holds(dequantize) -> bool:
    """Every code 0x38 (the value 1.0): the dequantised cache must be exactly
    the scale of each row's 64-token block, per (sequence, KV head), with a
    ragged last block (Tmax = 150: blocks of 64, 64 and 22 rows)."""
    B, G, Tmax, D = 2, 3, 150, 16
    codes = np.full((B, G, Tmax, D), 0x38, dtype=np.uint8)
    scales = (np.arange(B * G * 3, dtype=np.float32).reshape(B, G, 3) + 1.0) * np.float32(0.25)
    deq = dequantize(codes, scales)
    want = np.repeat(scales.astype(np.float64), 64, axis=2)[:, :, :Tmax, None]
    return deq.shape == codes.shape and bool(np.all(deq == want))


def test_dequantize_uses_each_64_token_blocks_own_scale():
    assert _block_scale_pin_holds(oracle.dequantize_fp8)


def test_block_scale_pin_catches_planted_mistakes():
    """Copies of the dequantiser with a plausible mistake fail the pin:
    32-token blocks, and the scale of the next KV head."""
    def blocks_of_32(codes, scales):
        B, G, Tmax, D = codes.shape
        sc = np.asarray(scales, dtype=np.float64)
        idx = np.minimum(np.arange(Tmax) // 32, sc.shape[2] - 1)
        return oracle.e4m3_to_f64(codes) * sc[:, :, idx, None]

    def next_head(codes, scales):
        return oracle.dequantize_fp8(codes, np.roll(scales, 1, axis=1))

    assert not _block_scale_pin_holds(blocks_of_32)
    assert not _block_scale_pin_holds(next_head)
