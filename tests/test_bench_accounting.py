"""The bench's accounting against numbers worked out by hand from the
definitions, so that a roofline fraction or a launch count cannot drift from
the workload it claims to measure.

- Bytes a decode step must move: the valid K and V, 2 x sum_b T_b x G x D x
  2 bytes (the KV-cache sizing of "GQA analysis", section "KV cache", summed
  over the batch), plus Q in and O out (bf16), LSE out (fp32) and the lengths
  (int32). The totals below are worked out per workload, not by the formula.
- FLOPs: 4 x sq x H x D per visible key (QK^T and PV); for a fresh prefill of
  n tokens each head sees n(n+1)/2 keys.
- Launches: one decode kernel per step; a prefill step adds a combine launch
  only when the library splits key ranges (short chunks on a mostly idle GPU).
- End to end: a step copies the cache rows each sequence holds, nothing more.
"""
import numpy as np
import pytest

import bench
import synthetic as syn

# (workload, algorithmic bytes per step), worked out by hand:
#   tiny: 2*1024*8*64*2 = 2,097,152 KV + 2*(32*64*2) Q,O + 32*4 LSE + 4
#   Llama layer: 2*16*4096*8*128*2 = 268,435,456 KV + 2*(16*32*128*2) + 16*32*4 + 64
#   MHA end: 2*8*4096*32*128*2 = 536,870,912 + 2*(8*32*128*2) + 8*32*4 + 32
#   MQA end: 2*64*8192*1*128*2 = 268,435,456 + 2*(64*32*128*2) + 64*32*4 + 256
#   long context B = 1: 2*131072*8*128*2 = 536,870,912 + 2*(64*128*2) + 64*4 + 4
#   long context B = 4: 4 x the KV of B = 1 + 2*(4*64*128*2) + 4*64*4 + 16
BYTES = {
    "tiny_gqa_d64": 2_097_152 + 8_192 + 128 + 4,
    "llama3_8b_layer": 268_435_456 + 262_144 + 2_048 + 64,
    "mha_end": 536_870_912 + 131_072 + 1_024 + 32,
    "mqa_end": 268_435_456 + 1_048_576 + 8_192 + 256,
    "long_ctx_b1": 536_870_912 + 32_768 + 256 + 4,
    "long_ctx_b4": 2_147_483_648 + 131_072 + 1_024 + 16,
}


@pytest.mark.parametrize("name", sorted(BYTES))
def test_decode_bytes_per_step(name):
    cfg = syn.config_by_name(name)
    lens = syn.seq_lens_for(cfg)
    assert bench.algorithmic_bytes(cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D, lens) == BYTES[name]


def test_decode_bytes_totals():
    """The sums above, written out: 2,105,476 (tiny), 268,699,712 (Llama
    layer), 537,003,040 (MHA end), 269,492,480 (MQA end), 536,903,940 and
    2,147,615,760 (long context)."""
    assert [BYTES[n] for n in ("tiny_gqa_d64", "llama3_8b_layer", "mha_end", "mqa_end",
                               "long_ctx_b1", "long_ctx_b4")] == [
        2_105_476, 268_699_712, 537_003_040, 269_492_480, 536_903_940, 2_147_615_760]


def test_decode_flops():
    # Llama layer: 4 * 1 * 32 * 128 * (16 * 4096) = 2^30
    cfg = syn.config_by_name("llama3_8b_layer")
    assert bench.algorithmic_flops(cfg.sq, cfg.H, cfg.D, syn.seq_lens_for(cfg)) == 1 << 30
    # MQA end: 4 * 32 * 128 * 64 * 8192 = 2^33
    cfg = syn.config_by_name("mqa_end")
    assert bench.algorithmic_flops(cfg.sq, cfg.H, cfg.D, syn.seq_lens_for(cfg)) == 1 << 33


def test_prefill_flops_causal_triangle():
    cfg = syn.config_by_name("prefill_llama3_8b_8k")     # fresh: T = sq = 8192
    n = 8192
    assert bench.visible_keys(cfg.sq, syn.seq_lens_for(cfg)) == n * (n + 1) // 2
    assert bench.prefill_flops(cfg.H, cfg.D, cfg.sq, syn.seq_lens_for(cfg)) == 4 * 32 * 128 * n * (n + 1) // 2
    # a 64-token chunk after 4032 cached tokens: token s sees 4033 + s keys
    cfg = syn.config_by_name("chunked_prefill_q64_d64")
    assert bench.visible_keys(cfg.sq, syn.seq_lens_for(cfg)) == sum(4033 + s for s in range(64))
    # decode's sq = 4 causal rows see T-3 .. T keys
    assert bench.visible_keys(4, [10, 2]) == (7 + 8 + 9 + 10) + (0 + 0 + 1 + 2)


def test_prefill_launches_per_step(monkeypatch):
    """152 SMs: the 64-token D = 64 chunk has 8 pairs of row tiles (B*G = 8,
    256 rows), so its 32 key tiles are split 16 ways and a combine follows;
    the three large prefills fill the GPU unsplit."""
    monkeypatch.delenv("GQA_PREFILL_SPLITS", raising=False)
    got = {c.name: bench.prefill_launches_per_step(c.B, c.sq, c.H, c.G, c.Tmax, 152)
           for c in syn.PREFILL_CONFIGS}
    assert got == {"chunked_prefill_q64_d64": 2, "prefill_d64_4k": 1, "prefill_llama3_8b_8k": 1,
                   "chunked_prefill_llama3_8b": 1}
    monkeypatch.setenv("GQA_PREFILL_SPLITS", "1")
    assert bench.prefill_launches_per_step(1, 64, 32, 8, 4096, 152) == 1
    monkeypatch.setenv("GQA_PREFILL_SPLITS", "4")
    assert bench.prefill_launches_per_step(4, 2048, 32, 8, 8192, 152) == 2


def test_percentiles():
    assert bench._percentiles_us([]) is None
    assert bench._percentiles_us([0.001 * i for i in range(1, 12)]) == pytest.approx([2.0, 6.0, 10.0])


@pytest.mark.parametrize("fp8", [False, True])
def test_e2e_copies_cover_exactly_the_valid_rows(fp8):
    """The end-to-end step copies every row a sequence holds (for fp8 block
    scales, every 64-token block its rows touch), each once, and nothing past
    a length; runs of full sequences are single copies."""
    import torch
    B, G, Tmax, D = 5, 3, 130, 4
    lens = np.array([130, 130, 7, 0, 130], dtype=np.int32)
    host = torch.arange(B * G * Tmax * D, dtype=torch.float32).view(B, G, Tmax, D)
    dev = torch.zeros_like(host)
    hkv, dkv = [host], [dev]
    if fp8:
        nb = -(-Tmax // 64)
        hkv.append(torch.arange(B * G * nb, dtype=torch.float32).view(B, G, nb) + 1)
        dkv.append(torch.zeros(B, G, nb))
    pairs = bench.e2e_copy_pairs(dkv, hkv, lens, fp8=fp8)
    for d, h in pairs:
        d.copy_(h)
    for b in range(B):
        n = int(lens[b])
        assert torch.equal(dev[b, :, :n], host[b, :, :n])
        assert not dev[b, :, n:].any()
        if fp8:
            nbk = -(-n // 64)
            assert torch.equal(dkv[1][b, :, :nbk], hkv[1][b, :, :nbk])
            assert not dkv[1][b, :, nbk:].any()
    full_runs = [p for p in pairs if p[1].dim() == host.dim() and p[1].shape[0] != G]
    assert [p[1].shape[0] for p in full_runs] == [2, 1]          # sequences 0-1, then 4
    copied = sum(h.numel() for _, h in pairs if h.dim() >= 2 and h.shape[-1] == D)   # K/V, not scales
    assert copied == int(lens.sum()) * G * D
