"""Pins for the CPU oracle: each check ties the oracle to something that does not
come from the oracle itself -- the head-mapping table the first page prints,
the repeat_kv / repeat_interleave expansions the first page describes, PyTorch's
scaled_dot_product_attention (float64, enable_gqa) as a library routine,
high-precision brute force on tiny inputs, and closed forms (a single key, equal
keys, a dominant key, value shifts, empty rows, causal visibility).

Every pin takes an `orc` (an oracle.Oracle) so that the same checks can be run
against deliberately broken copies of the oracle (tests/test_oracle_mutants.py)
to show that a plausible mistake fails at least one of them.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NAN = syn.BF16_NAN


def _f64(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def _bits(x):
    return syn.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def make_case(B, sq, H, G, D, Tmax, lens, seed, tail=NAN):
    lens = np.asarray(lens, dtype=np.int32)
    q = syn.normal_bf16(seed, syn.STREAM_Q, (B, sq, H, D))
    k = syn.fill_cache(seed, syn.STREAM_K, B, G, Tmax, D, lens, tail, threads=1)
    v = syn.fill_cache(seed, syn.STREAM_V, B, G, Tmax, D, lens, tail, threads=1)
    return q, k, v, lens


def load_mapping_table():
    """{query head: KV head} from the printed Exaone4 table (32 -> 8)."""
    table = {}
    with open(os.path.join(GOLDEN, "head_mapping_exaone4_h32_g8.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            heads, kv = line.split()
            for h in heads.split(","):
                table[int(h)] = int(kv)
    return table


# ---------------------------------------------------------------- head mapping

def pin_mapping_page_table(orc):
    """V of KV head g is the constant g+1, so out[h] must be kv(h)+1 with kv(h)
    read from the page's printed table (query heads 0..31 -> KV heads 0..7)."""
    table = load_mapping_table()
    assert sorted(table) == list(range(32))
    H, G, D, T = 32, 8, 8, 5
    q = syn.normal_bf16(11, 1, (1, 1, H, D))
    k = syn.normal_bf16(11, 2, (1, G, T, D))
    v = np.empty((1, G, T, D), dtype=np.uint16)
    for g in range(G):
        v[0, g] = _bits(g + 1.0)
    out, lse = orc.gqa_decode(q, k, v, [T], 1 / math.sqrt(D))
    for h in range(H):
        np.testing.assert_allclose(out[0, 0, h], table[h] + 1.0, rtol=1e-12, atol=0)
    assert np.all(np.isfinite(lse))


def pin_mapping_repeat_semantics(orc):
    """For other (H, G): the KV head each query head reads must be the one that
    np.repeat(arange(G), H/G) -- the layout repeat_kv / repeat_interleave build
    -- puts at that head position."""
    for H, G in [(8, 1), (8, 2), (8, 4), (8, 8), (12, 3), (6, 2), (64, 8)]:
        D, T = 4, 3
        q = syn.normal_bf16(12, 1, (1, 1, H, D))
        k = syn.normal_bf16(12, 2, (1, G, T, D))
        v = np.empty((1, G, T, D), dtype=np.uint16)
        for g in range(G):
            v[0, g] = _bits(g + 1.0)
        out, _ = orc.gqa_decode(q, k, v, [T], 0.5)
        kv_of_head = np.repeat(np.arange(G), H // G)
        for h in range(H):
            np.testing.assert_allclose(out[0, 0, h], kv_of_head[h] + 1.0, rtol=1e-12, atol=0)


# ------------------------------------------------- expansion == no expansion

def _expand_reshape(x, n_rep):
    """Hugging Face repeat_kv as the first page describes it: a stride-0 expand
    over a new repeat axis, then a reshape that copies into H heads."""
    B, G, T, D = x.shape
    view = np.broadcast_to(x[:, :, None, :, :], (B, G, n_rep, T, D))
    return np.ascontiguousarray(view.reshape(B, G * n_rep, T, D))


def pin_repeat_kv_expand_reshape(orc):
    """GQA on the G-head cache equals per-head MHA (G = H) on the repeat_kv
    expanded cache, bit for bit (same values, same per-row loop order)."""
    for (B, sq, H, G, D, Tmax, lens) in [(2, 1, 8, 2, 16, 12, [12, 7]),
                                         (2, 3, 12, 3, 8, 10, [10, 5]),
                                         (1, 2, 4, 1, 8, 6, [6])]:
        q, k, v, lens = make_case(B, sq, H, G, D, Tmax, lens, seed=13)
        n_rep = H // G
        a_out, a_lse = orc.gqa_decode(q, k, v, lens, 1 / math.sqrt(D))
        b_out, b_lse = orc.gqa_decode(q, _expand_reshape(k, n_rep), _expand_reshape(v, n_rep),
                                      lens, 1 / math.sqrt(D))
        assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)


def pin_repeat_interleave(orc):
    """Same with torch.repeat_interleave(H/G, dim=head), the reference semantics
    the first page quotes for scaled_dot_product_attention(enable_gqa=True)."""
    B, sq, H, G, D, Tmax = 2, 2, 8, 4, 8, 9
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [9, 4], seed=14)
    n_rep = H // G
    ki = torch.from_numpy(k.astype(np.int32)).repeat_interleave(n_rep, dim=1)
    vi = torch.from_numpy(v.astype(np.int32)).repeat_interleave(n_rep, dim=1)
    a_out, a_lse = orc.gqa_decode(q, k, v, lens, 0.3)
    b_out, b_lse = orc.gqa_decode(q, ki.numpy().astype(np.uint16), vi.numpy().astype(np.uint16),
                                  lens, 0.3)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)


# -------------------------------------------------- a library routine: SDPA

def sdpa_reference(q, k, v, lens, scale=None):
    """torch scaled_dot_product_attention in float64 on the CPU, enable_gqa=True,
    one sequence at a time over its valid keys, with an explicit bottom-right
    causal mask among the sq new tokens. Also returns the natural-log LSE from
    torch.logsumexp over the same masked, scaled scores."""
    B, sq, H, D = q.shape
    G = k.shape[1]
    out = np.zeros((B, sq, H, D))
    lse = np.zeros((B, sq, H))
    for b in range(B):
        T = int(lens[b])
        qb = torch.from_numpy(_f64(q[b])).permute(1, 0, 2).unsqueeze(0)  # [1,H,sq,D]
        kb = torch.from_numpy(_f64(k[b, :, :T])).unsqueeze(0)            # [1,G,T,D]
        vb = torch.from_numpy(_f64(v[b, :, :T])).unsqueeze(0)
        pos = torch.arange(T)
        allowed = pos[None, :] <= (T - sq + torch.arange(sq))[:, None]   # [sq,T]
        kw = {} if scale is None else {"scale": scale}
        ob = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, attn_mask=allowed, enable_gqa=True, **kw)
        out[b] = ob[0].permute(1, 0, 2).numpy()
        s = scale if scale is not None else 1 / math.sqrt(D)
        krep = kb.repeat_interleave(H // G, dim=1)
        scores = (qb @ krep.transpose(-1, -2)) * s
        scores = scores.masked_fill(~allowed, float("-inf"))
        lse[b] = torch.logsumexp(scores, dim=-1)[0].permute(1, 0).numpy()
    return out, lse


def pin_sdpa_float64(orc):
    """Agreement with PyTorch's own attention (float64, default scale 1/sqrt(D),
    which also pins the sqrt reading of the scale) across GQA, the MHA end
    (G = H), the MQA end (G = 1), ragged lengths and sq = 4 causal rows."""
    cases = [(2, 1, 8, 2, 16, 40, [40, 23]),
             (1, 1, 8, 8, 8, 17, [17]),        # MHA end
             (3, 1, 8, 1, 8, 19, [19, 1, 8]),  # MQA end
             (2, 4, 8, 2, 16, 33, [33, 6]),    # causal among 4 new tokens
             (1, 2, 6, 3, 4, 5, [5])]
    for (B, sq, H, G, D, Tmax, lens) in cases:
        q, k, v, lens = make_case(B, sq, H, G, D, Tmax, lens, seed=15)
        out, lse = orc.gqa_decode(q, k, v, lens, 1 / math.sqrt(D))
        ref_out, ref_lse = sdpa_reference(q, k, v, lens)
        np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


# ------------------------------------------------------ brute force, tiny

def pin_bruteforce_mpmath(orc):
    """40-digit brute force of the definition with no max subtraction:
    w_t = exp(x_t), out = sum w_t v_t / sum w_t, lse = log sum w_t."""
    import mpmath
    mpmath.mp.dps = 40
    B, sq, H, G, D, Tmax = 1, 2, 4, 2, 3, 6
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [6], seed=16)
    scale = 0.7
    out, lse = orc.gqa_decode(q, k, v, lens, scale)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    for s in range(sq):
        for h in range(H):
            g = [0, 0, 1, 1][h]  # H=4, G=2: heads {0,1} -> 0, {2,3} -> 1
            n = int(lens[0]) - sq + s + 1
            xs = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(qf[0, s, h, d]) * mpmath.mpf(kf[0, g, t, d])
                                                  for d in range(D)) for t in range(n)]
            ws = [mpmath.exp(x) for x in xs]
            Z = mpmath.fsum(ws)
            for d in range(D):
                ref = mpmath.fsum(w * mpmath.mpf(vf[0, g, t, d]) for t, w in enumerate(ws)) / Z
                assert abs(out[0, s, h, d] - float(ref)) <= 1e-14 * max(1.0, abs(float(ref)))
            assert abs(lse[0, s, h] - float(mpmath.log(Z))) <= 1e-14 * max(1.0, abs(float(mpmath.log(Z))))


# ----------------------------------------------------------- closed forms

def pin_single_key(orc):
    """One visible key: the softmax weight is exactly 1, so out == v[0] bit for
    bit and lse == the scaled score x_0."""
    D = 16
    q = syn.normal_bf16(17, 1, (1, 1, 4, D))
    k = syn.normal_bf16(17, 2, (1, 2, 3, D))
    v = syn.normal_bf16(17, 3, (1, 2, 3, D))
    out, lse = orc.gqa_decode(q, k, v, [1], 0.25)
    for h in range(4):
        g = h // 2
        assert np.array_equal(out[0, 0, h], _f64(v[0, g, 0]))
        x0 = 0.25 * float(np.dot(_f64(q[0, 0, h]), _f64(k[0, g, 0])))
        assert abs(lse[0, 0, h] - x0) <= 1e-14 * max(1.0, abs(x0))


def pin_equal_keys(orc):
    """All visible keys equal: the softmax is uniform, out = mean of the visible
    V rows and lse = x + ln(n)."""
    for sq in (1, 3):
        B, H, G, D, Tmax = 1, 4, 2, 8, 11
        q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [11], seed=18)
        k[:, :, :, :] = k[:, :, :1, :]
        out, lse = orc.gqa_decode(q, k, v, lens, 0.4)
        for s in range(sq):
            n = 11 - sq + s + 1
            for h in range(H):
                g = h // 2
                np.testing.assert_allclose(out[0, s, h], _f64(v[0, g, :n]).mean(axis=0),
                                           rtol=0, atol=1e-14)
                x = 0.4 * float(np.dot(_f64(q[0, s, h]), _f64(k[0, g, 0])))
                assert abs(lse[0, s, h] - (x + math.log(n))) <= 1e-13


def pin_dominant_key(orc):
    """One key whose score beats every other by > 100: out is that key's V row
    and lse its score, to double precision."""
    D, T = 8, 9
    for tstar in (0, 4, 8):
        q = np.full((1, 1, 2, D), _bits(8.0), dtype=np.uint16)
        k = syn.normal_bf16(19 + tstar, 2, (1, 1, T, D))
        v = syn.normal_bf16(19 + tstar, 3, (1, 1, T, D))
        k[0, 0, tstar] = _bits(8.0)
        out, lse = orc.gqa_decode(q, k, v, [T], 1 / math.sqrt(D))
        xstar = 8.0 * 8.0 * D / math.sqrt(D)
        for h in range(2):
            np.testing.assert_allclose(out[0, 0, h], _f64(v[0, 0, tstar]), rtol=1e-15, atol=0)
            assert abs(lse[0, 0, h] - xstar) <= 1e-12


def pin_value_shift(orc):
    """Softmax weights sum to one: adding a constant c to every V row shifts out
    by exactly c (integer-valued V so that V + c is exact in bf16)."""
    B, sq, H, G, D, Tmax = 2, 2, 4, 2, 8, 13
    q, k, _, lens = make_case(B, sq, H, G, D, Tmax, [13, 8], seed=20, tail=0)
    ints = syn.uniform_int(20, 9, B * G * Tmax * D, -8, 8).reshape(B, G, Tmax, D)
    v = _bits(ints.astype(np.float32))
    v3 = _bits((ints + 3).astype(np.float32))
    out, _ = orc.gqa_decode(q, k, v, lens, 0.35)
    out3, _ = orc.gqa_decode(q, k, v3, lens, 0.35)
    np.testing.assert_allclose(out3, out + 3.0, rtol=0, atol=1e-13)


def pin_token_permutation(orc):
    """Attention has no notion of order beyond the mask: permuting the visible
    tokens (K and V rows together) leaves out and lse unchanged."""
    B, sq, H, G, D, Tmax = 1, 1, 4, 2, 8, 15
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [15], seed=21)
    perm = np.random.default_rng(0).permutation(15)
    out, lse = orc.gqa_decode(q, k, v, lens, 0.3)
    out_p, lse_p = orc.gqa_decode(q, k[:, :, perm], v[:, :, perm], lens, 0.3)
    np.testing.assert_allclose(out_p, out, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse_p, lse, rtol=0, atol=1e-14)


def pin_lse_normalisation(orc):
    """lse is the log of the softmax denominator: sum_t exp(x_t - lse) = 1 and
    out = sum_t exp(x_t - lse) v_t, with the scores x_t from a numpy matmul."""
    B, sq, H, G, D, Tmax = 1, 1, 6, 3, 16, 21
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [21], seed=22)
    out, lse = orc.gqa_decode(q, k, v, lens, 0.25)
    for h in range(H):
        g = h // 2
        x = 0.25 * (_f64(k[0, g]) @ _f64(q[0, 0, h]))
        w = np.exp(x - lse[0, 0, h])
        assert abs(w.sum() - 1.0) <= 1e-13
        np.testing.assert_allclose(w @ _f64(v[0, g]), out[0, 0, h], rtol=0, atol=1e-13)


# -------------------------------------------------- causal visibility, edges

def pin_causal_prefix(orc):
    """Row s of an sq = 4 call equals a one-token call whose length stops at that
    token's own position (T_b - sq + s + 1), bit for bit."""
    B, sq, H, G, D, Tmax = 3, 4, 4, 2, 8, 20
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [20, 9, 4], seed=23)
    out, lse = orc.gqa_decode(q, k, v, lens, 0.3)
    for b in range(B):
        for s in range(sq):
            o1, l1 = orc.gqa_decode(q[b:b + 1, s:s + 1], k[b:b + 1], v[b:b + 1],
                                    [int(lens[b]) - sq + s + 1], 0.3)
            assert np.array_equal(o1[0, 0], out[b, s]) and np.array_equal(l1[0, 0], lse[b, s])


def pin_visibility_boundary(orc):
    """Poison the cache row at position T - sq + s' (NaN in K and V): rows s < s'
    must stay finite and rows s >= s' must see it (become NaN)."""
    B, sq, H, G, D, Tmax, T = 1, 4, 2, 1, 8, 12, 10
    base = make_case(B, sq, H, G, D, Tmax, [T], seed=24)
    for sp in range(sq):
        q, k, v, lens = (x.copy() for x in base)
        p = T - sq + sp
        k[0, 0, p] = NAN
        v[0, 0, p] = NAN
        out, _ = orc.gqa_decode(q, k, v, lens, 0.3)
        for s in range(sq):
            finite = bool(np.all(np.isfinite(out[0, s])))
            assert finite == (s < sp), (sp, s)


def pin_tail_unread(orc):
    """Entries at t >= seq_lens[b] are NaN; the result must not see them."""
    q, k, v, lens = make_case(3, 2, 8, 2, 8, 30, [30, 2, 17], seed=25)
    out, lse = orc.gqa_decode(q, k, v, lens, 0.3)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def pin_empty_rows(orc):
    """A row with no visible key (T_b - sq + s < 0) gets out = 0, lse = -inf; the
    first visible row of a short sequence sees exactly one key."""
    B, sq, H, G, D, Tmax = 2, 3, 2, 1, 4, 6
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [0, 2], seed=26)
    out, lse = orc.gqa_decode(q, k, v, lens, 0.5)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(out[1, 0] == 0) and np.all(np.isneginf(lse[1, 0]))
    for h in range(H):
        assert np.array_equal(out[1, 1, h], _f64(v[1, 0, 0]))
    assert np.all(np.isfinite(out[1, 2])) and np.all(np.isfinite(lse[1, 2]))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
