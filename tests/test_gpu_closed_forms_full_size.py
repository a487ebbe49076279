"""Closed forms at the decode workloads' full sizes, in the launch configuration
the bench times, checked on EVERY output row (the full-size oracle tests
compare a sample of rows; these need no oracle). The attention definition
(softmax of the scaled scores against the KV head g(h) = h / (H/G), times V;
"GQA analysis", section "Grouped broadcast") fixes both:

- One dominant key per KV head. Keys are N(0,1) except one row t*(b, g),
  visible to every new token, set to 4 in every dimension. Query rows are
  constant: 1 + j/8 in every dimension for head j of its group. The dominant
  score x* = scale * D * 4 * (1 + j/8) beats every other by more than 30
  (checked below from the keys), so the softmax weight off t* sums to less
  than 1e-9: out = V[t*] (values of order 1, where the 1e-2 bar is strict) and
  lse = x*; the kernel's output must round to V[t*] itself. The CTA shares
  that do not hold t* give partials whose maximum lies tens below the
  unit's, which the combine must weigh out; heads of different groups see
  different t*, so a wrong g(h) fails too.
- Equal keys. Every visible key of unit (b, g) is the same row, so each query
  row's scores are all equal: out = the mean of V over its visible keys and
  lse = x + ln(number of visible keys). A partial that the combine dropped,
  counted twice or weighed wrongly moves lse by ln(1 +- its share of keys).

Cache rows past each sequence's length hold NaN, as in every parity test.
"""
import math

import numpy as np
import pytest
import torch

import synthetic as syn
from gpu_helpers import compare, note_quality, run_gpu

pytestmark = pytest.mark.gpu

NAMES = ["llama3_8b_layer", "mqa_end", "long_ctx_b1", "long_ctx_b4", "ragged_sq4"]
FOUR = int(syn.f32_to_bf16_bits(np.float32(4.0))[0])


def _f64(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def _done():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", NAMES)
def test_dominant_key_every_row(name):
    cfg = syn.config_by_name(name)
    _, k, v, lens = syn.make_inputs(cfg)
    B, sq, H, G, D = cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D
    hpg = H // G
    j = np.arange(H) % hpg
    q = np.empty((B, sq, H, D), dtype=np.uint16)
    q[...] = syn.f32_to_bf16_bits((1.0 + j / 8.0).astype(np.float32))[None, None, :, None]

    rng = np.random.default_rng(cfg.seed + 11)
    vstar = np.empty((B, G, D))
    worst = 0.0   # largest bound on the weight off t*, over every row
    for b in range(B):
        T = int(lens[b])
        for g in range(G):
            ts = int(rng.integers(0, T - sq + 1))      # visible to every new token
            k[b, g, ts] = FOUR
            vstar[b, g] = _f64(v[b, g, ts])
            rowsum = syn.bf16_bits_to_f32(k[b, g, :T]).sum(axis=1, dtype=np.float64)
            rowsum[ts] = -np.inf
            # smallest gap x* - x_t is at j = 0 (multiplier 1); at most T keys
            gap = cfg.scale * (4.0 * D - rowsum.max())
            worst = max(worst, T * math.exp(-gap))
    assert worst < 1e-9, f"{name}: keys leave weight {worst:.2e} off the dominant key"

    out, lse = run_gpu(q, k, v, lens, cfg.scale)
    ref_out = np.broadcast_to(np.repeat(vstar, hpg, axis=1)[:, None], (B, sq, H, D))
    xstar = cfg.scale * D * 4.0 * (1.0 + j / 8.0)
    ref_lse = np.broadcast_to(xstar[None, None, :], (B, sq, H))
    err, _ = compare(out, lse, ref_out, ref_lse, what=f"{name} dominant key")
    note_quality(f"{name} dominant key (every row)", err, ref_out)
    # Stricter than the bar: V[t*] is a bf16 value and the weight off t* is
    # below 1e-9, so the fp32 result rounds back to V[t*] itself; allow one
    # bf16 step (2^-7 |x|), and 1e-6 where V[t*] is near zero.
    step = np.abs(ref_out) * 2.0 ** -7 + 1e-6
    assert np.all(np.abs(out - ref_out) <= step), f"{name}: dominant key off by more than one bf16 step"
    _done()


@pytest.mark.parametrize("name", NAMES)
def test_equal_keys_every_row(name):
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg)
    B, sq, H, G, D = cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D
    hpg = H // G
    ref_out = np.empty((B, sq, H, D))
    ref_lse = np.empty((B, sq, H))
    qf = _f64(q)
    for b in range(B):
        T = int(lens[b])
        k[b, :, :T] = k[b, :, :1]
        for g in range(G):
            vf = _f64(v[b, g, :T])
            acc = vf[:T - sq + 1].sum(axis=0)
            k0 = _f64(k[b, g, 0])
            for s in range(sq):
                n = T - sq + s + 1                     # keys visible to new token s
                if s:
                    acc = acc + vf[n - 1]
                heads = slice(g * hpg, (g + 1) * hpg)
                ref_out[b, s, heads] = acc / n
                ref_lse[b, s, heads] = cfg.scale * (qf[b, s, heads] @ k0) + math.log(n)

    out, lse = run_gpu(q, k, v, lens, cfg.scale)
    err, _ = compare(out, lse, ref_out, ref_lse, what=f"{name} equal keys")
    note_quality(f"{name} equal keys (every row)", err, ref_out)
    _done()



# ---------------------------------------------------------------- fp8 cache
# The same two forms over an e4m3 cache with one scale per 64-token block,
# against the dequantised values (torch's e4m3 decoding of the codes times
# the block's scale). On one row tile the fp8 kernel runs two groups of
# consumer warps on alternate tiles, whose states merge in shared memory
# before the cross-CTA merge: a dominant key sits in one group's state only.
# The kernel carries V's scale as an fp16 multiplier of P, so the output is
# checked against the bar only (no one-step bound).

FP8_NAMES = ["llama3_8b_layer", "mqa_end", "long_ctx_b1"]


def _dequant_unit(codes, scales, b, g, T):
    x = torch.from_numpy(np.ascontiguousarray(codes[b, g, :T])).view(torch.float8_e4m3fn).double()
    s = torch.from_numpy(scales[b, g]).double().repeat_interleave(64)[:T, None]
    return (x * s).numpy()


def _run_fp8(cfg, q, kc, ks, vc, vs, lens):
    import grouped_query_decode_gb300 as gq
    from gpu_helpers import bf16_to_f64, to_device_bf16
    out = torch.empty(cfg.B, cfg.sq, cfg.H, cfg.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(cfg.B, cfg.sq, cfg.H, dtype=torch.float32, device="cuda")
    gq.gqa_decode_fp8(to_device_bf16(q), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                      torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(),
                      torch.from_numpy(lens).cuda(), cfg.scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", FP8_NAMES)
def test_fp8_dominant_key_every_row(name):
    cfg = syn.config_by_name(name)
    _, k, v, lens = syn.make_inputs(cfg)
    B, sq, H, G, D = cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D
    hpg = H // G
    j = np.arange(H) % hpg
    mult = 1.0 + j / 8.0
    q = np.empty((B, sq, H, D), dtype=np.uint16)
    q[...] = syn.f32_to_bf16_bits(mult.astype(np.float32))[None, None, :, None]
    rng = np.random.default_rng(cfg.seed + 12)
    tstar = np.empty((B, G), dtype=np.int64)
    for b in range(B):
        for g in range(G):
            tstar[b, g] = int(rng.integers(0, int(lens[b]) - sq + 1))
            k[b, g, tstar[b, g]] = FOUR
    kc, ks = syn.fp8_cache(k, lens)
    vc, vs = syn.fp8_cache(v, lens)
    del k, v

    ref_out = np.empty((B, sq, H, D))
    ref_lse = np.empty((B, sq, H))
    worst = 0.0
    for b in range(B):
        T = int(lens[b])
        for g in range(G):
            ts = int(tstar[b, g])
            rowsum = _dequant_unit(kc, ks, b, g, T).sum(axis=1)
            xs = rowsum[ts]
            rowsum[ts] = -np.inf
            worst = max(worst, T * math.exp(-cfg.scale * (xs - rowsum.max())))
            heads = slice(g * hpg, (g + 1) * hpg)
            ref_out[b, :, heads] = _dequant_unit(vc, vs, b, g, ts + 1)[ts]
            ref_lse[b, :, heads] = cfg.scale * xs * mult[heads]
    assert worst < 1e-9, f"{name}: keys leave weight {worst:.2e} off the dominant key"

    out, lse = _run_fp8(cfg, q, kc, ks, vc, vs, lens)
    err, _ = compare(out, lse, ref_out, ref_lse, what=f"{name} fp8 dominant key")
    note_quality(f"{name} fp8 dominant key (every row)", err, ref_out)
    _done()


@pytest.mark.parametrize("name", FP8_NAMES)
def test_fp8_equal_keys_every_row(name):
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg)
    B, sq, H, G, D = cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D
    hpg = H // G
    for b in range(B):
        k[b, :, :int(lens[b])] = k[b, :, :1]
    kc, ks = syn.fp8_cache(k, lens)
    vc, vs = syn.fp8_cache(v, lens)
    del k, v
    qf = _f64(q)
    ref_out = np.empty((B, sq, H, D))
    ref_lse = np.empty((B, sq, H))
    for b in range(B):
        T = int(lens[b])
        for g in range(G):
            kd = _dequant_unit(kc, ks, b, g, T)
            assert np.array_equal(kd, np.broadcast_to(kd[:1], kd.shape)), "dequantised keys differ"
            vd = _dequant_unit(vc, vs, b, g, T)
            heads = slice(g * hpg, (g + 1) * hpg)
            for s in range(sq):
                n = T - sq + s + 1
                ref_out[b, s, heads] = vd[:n].mean(axis=0)
                ref_lse[b, s, heads] = cfg.scale * (qf[b, s, heads] @ kd[0]) + math.log(n)

    out, lse = _run_fp8(cfg, q, kc, ks, vc, vs, lens)
    err, _ = compare(out, lse, ref_out, ref_lse, what=f"{name} fp8 equal keys")
    note_quality(f"{name} fp8 equal keys (every row)", err, ref_out)
    _done()


# ------------------------------------------------- periodic keys (causal edge)
# Key t is 32 e_(t mod D) (one-hot), and the query of new token s of head j is
# 32 (1 + j/8) e_(p mod D), p = T - sq + s its position. A key scores
# x = 1024 scale (1 + j/8) (90 or more here) when t = p mod D and exactly 0
# otherwise, so out = the mean of V over the visible keys t <= p with
# t = p (mod D), and lse = x + ln(their number). The diagonal key (t = p)
# is always among them and the next key of the class (p + D) never: any
# causal off-by-one moves the result. Rows whose first tiles hold no
# matching key also take the rescale path when the first one arrives.

def _periodic_case(cfg):
    _, _, v, lens = syn.make_inputs(cfg)
    B, sq, H, G, D, Tmax = cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D, cfg.Tmax
    hpg = H // G
    mult = 1.0 + (np.arange(H) % hpg) / 8.0
    k = np.full((B, G, Tmax, D), syn.BF16_NAN, dtype=np.uint16)
    q = np.zeros((B, sq, H, D), dtype=np.uint16)
    ref_out = np.empty((B, sq, H, D))
    ref_lse = np.empty((B, sq, H))
    x = 1024.0 * cfg.scale * mult
    qvals = syn.f32_to_bf16_bits((32.0 * mult).astype(np.float32))
    for b in range(B):
        T = int(lens[b])
        t = np.arange(T)
        k[b, :, :T] = 0
        k[b, :, t, t % D] = int(syn.f32_to_bf16_bits(np.float32(32.0))[0])
        p = T - sq + np.arange(sq)                     # positions of the new tokens
        q[b, np.arange(sq)[:, None], np.arange(H)[None, :], (p % D)[:, None]] = qvals[None, :]
        count = p // D + 1
        Tp = -(-T // D) * D
        for g in range(G):
            vf = np.zeros((Tp, D))
            vf[:T] = _f64(v[b, g, :T])
            csum = np.cumsum(vf.reshape(Tp // D, D, D), axis=0)   # [row block, residue, dim]
            means = csum[p // D, p % D] / count[:, None]          # [sq, D]
            heads = slice(g * hpg, (g + 1) * hpg)
            ref_out[b, :, heads] = means[:, None, :]
            ref_lse[b, :, heads] = x[None, heads] + np.log(count)[:, None]
    return q, k, v, lens, ref_out, ref_lse


@pytest.mark.parametrize("name", NAMES + [c.name for c in syn.PREFILL_CONFIGS])
def test_periodic_keys_every_row(name):
    import grouped_query_decode_gb300 as gq
    cfg = syn.config_by_name(name)
    q, k, v, lens, ref_out, ref_lse = _periodic_case(cfg)
    entry = gq.gqa_prefill if cfg.rows > 32 else gq.gqa_decode
    out, lse = run_gpu(q, k, v, lens, cfg.scale, entry=entry)
    err, _ = compare(out, lse, ref_out, ref_lse, what=f"{name} periodic keys")
    note_quality(f"{name} periodic keys (every row)", err, ref_out)
    _done()
