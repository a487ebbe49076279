"""Pins for the oracle's cache append (CPU only): "GQA analysis", sections
"Projection and RoPE" and "Incremental decode" append the new token's K and V
to the caches and then attend over the whole cache, the new token included."""
import math

import numpy as np

import oracle
import synthetic as syn
from oracle_pins import _bits, _f64, make_case


def _placement_pin_holds(append) -> bool:
    """Exactly the sq positions that end at T_b (those >= 0) change, in order,
    and nothing else: worked out by hand for T = 12, 5, 1 and sq = 2."""
    B, sq, H, G, D, Tmax = 3, 2, 4, 2, 8, 12
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [12, 5, 1], seed=50)
    kn = syn.normal_bf16(51, 1, (B, sq, G, D))
    vn = syn.normal_bf16(51, 2, (B, sq, G, D))
    k2, v2 = append(k, v, kn, vn, lens)
    changed = np.zeros((B, Tmax), dtype=bool)
    for b in range(B):
        for t in range(Tmax):
            if not (np.array_equal(k2[b, :, t], k[b, :, t]) and np.array_equal(v2[b, :, t], v[b, :, t])):
                changed[b, t] = True
    return (changed[0].nonzero()[0].tolist() == [10, 11] and changed[1].nonzero()[0].tolist() == [3, 4]
            and changed[2].nonzero()[0].tolist() == [0]
            and np.array_equal(k2[1, :, 3], kn[1, 0]) and np.array_equal(v2[1, :, 4], vn[1, 1])
            and np.array_equal(k2[2, :, 0], kn[2, 1]) and np.array_equal(v2[2, :, 0], vn[2, 1]))


def test_new_rows_land_before_the_length_and_nothing_else_moves():
    assert _placement_pin_holds(oracle.append_f64)


def test_placement_pin_catches_planted_mistakes():
    """Copies of the append with a plausible mistake fail the pin: one slot
    late, the new tokens in reverse order, and K and V swapped."""
    def make(pos, order=lambda s, sq: s, swap=False):
        def append(k_cache, v_cache, k_new, v_new, seq_lens):
            k = np.array(k_cache, copy=True)
            v = np.array(v_cache, copy=True)
            B, G, Tmax, D = k.shape
            sq = k_new.shape[1]
            for b in range(B):
                for s in range(sq):
                    t = pos(int(seq_lens[b]), sq, s)
                    if 0 <= t < Tmax:
                        src = order(s, sq)
                        k[b, :, t, :] = (v_new if swap else k_new)[b, src]
                        v[b, :, t, :] = (k_new if swap else v_new)[b, src]
            return k, v
        return append

    assert _placement_pin_holds(make(lambda T, sq, s: T - sq + s))            # the right one
    assert not _placement_pin_holds(make(lambda T, sq, s: T - sq + s + 1))
    assert not _placement_pin_holds(make(lambda T, sq, s: T - sq + s, order=lambda s, sq: sq - 1 - s))
    assert not _placement_pin_holds(make(lambda T, sq, s: T - sq + s, swap=True))


def test_a_new_token_attends_to_itself():
    """One new token whose own key dominates its query: after the append the
    output is its own value row (the token sees itself, at position T - 1)."""
    D, T = 8, 9
    q = np.full((1, 1, 2, D), _bits(4.0), dtype=np.uint16)
    _, k, v, lens = make_case(1, 1, 2, 1, D, T, [T], seed=52)
    kn = np.full((1, 1, 1, D), _bits(4.0), dtype=np.uint16)
    vn = syn.normal_bf16(53, 1, (1, 1, 1, D))
    out, lse, _, _ = oracle.gqa_decode_append_f64(q, k, v, kn, vn, lens, 1 / math.sqrt(D))
    for h in range(2):
        np.testing.assert_allclose(out[0, 0, h], _f64(vn[0, 0, 0]), rtol=1e-12, atol=0)


def test_new_tokens_see_only_earlier_new_tokens():
    """sq = 4 new tokens; make new key s' dominant for every query: rows
    s >= s' return v_new[s'], rows s < s' cannot see it."""
    D, T, sq = 8, 10, 4
    for sp in range(sq):
        q = np.full((1, sq, 2, D), _bits(4.0), dtype=np.uint16)
        _, k, v, lens = make_case(1, sq, 2, 1, D, T, [T], seed=54)
        kn = syn.normal_bf16(55, 1, (1, sq, 1, D))
        kn[0, sp, 0] = _bits(4.0)
        vn = syn.normal_bf16(55, 2, (1, sq, 1, D))
        out, _, _, _ = oracle.gqa_decode_append_f64(q, k, v, kn, vn, lens, 1 / math.sqrt(D))
        for s in range(sq):
            hit = np.allclose(out[0, s, 0], _f64(vn[0, sp, 0]), rtol=1e-9, atol=0)
            assert hit == (s >= sp), (sp, s)


def test_append_then_attend_equals_attending_a_cache_built_with_the_rows():
    B, sq, H, G, D, Tmax = 2, 3, 8, 2, 16, 40
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [40, 17], seed=56)
    kn = syn.normal_bf16(57, 1, (B, sq, G, D))
    vn = syn.normal_bf16(57, 2, (B, sq, G, D))
    out, lse, k2, v2 = oracle.gqa_decode_append_f64(q, k, v, kn, vn, lens, 0.25)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k2, v2, lens, 0.25)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
