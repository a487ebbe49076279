"""The decode workloads at their full sizes, in the launch configuration the
bench times (default plan). The oracle recomputes a seeded sample of rows one
by one (first and last rows included); every row is checked for properties
that hold at any size: finite output and LSE, and each output element inside
the range of the V column it averages (softmax weights are non-negative and
sum to one)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_helpers import OUT_ATOL, compare, note_quality, run_gpu, to_device_bf16

pytestmark = pytest.mark.gpu

BIG = [c.name for c in syn.CONFIGS if c.name != "tiny_gqa_d64"]
SAMPLE_ROWS = 40


@pytest.mark.parametrize("name", BIG)
def test_full_size_workload(name):
    cfg = syn.config_by_name(name)
    q, k, v, lens = syn.make_inputs(cfg)          # NaN past each sequence's length
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    dl = torch.from_numpy(lens).cuda()
    out, lse = run_gpu(q, k, v, lens, cfg.scale, device_inputs=(dq, dk, dv, dl))

    # sampled rows against the oracle
    nrows = cfg.B * cfg.sq * cfg.H
    rng = np.random.default_rng(cfg.seed)
    rows = np.unique(np.concatenate([[0, nrows - 1], rng.choice(nrows, SAMPLE_ROWS, replace=False)]))
    ref_out = np.full((nrows, cfg.D), np.nan)
    ref_lse = np.full(nrows, np.nan)
    orc = oracle.get()
    for r in rows:
        o, l = orc.gqa_decode(q, k, v, lens, cfg.scale, rows=(int(r), int(r) + 1))
        ref_out[r] = o.reshape(nrows, cfg.D)[r]
        ref_lse[r] = l.reshape(nrows)[r]
    err, lerr = compare(out, lse, ref_out, ref_lse, rows=rows, what=name)
    print(f"{name}: sampled max-abs err out {err:.2e} lse {lerr:.2e}")
    note_quality(f"{name} ({len(rows)} sampled rows)", err, ref_out[rows])

    # every row: finite, and inside the per-column range of V over visible keys
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    o = torch.from_numpy(out).cuda()
    hpg = cfg.H // cfg.G
    for b in range(cfg.B):
        T = int(lens[b])
        vb = dv[b, :, :T].float()                        # [G, T, D]
        lo = vb.amin(dim=1).repeat_interleave(hpg, dim=0)  # [H, D]
        hi = vb.amax(dim=1).repeat_interleave(hpg, dim=0)
        ob = o[b].float()                                # [sq, H, D]
        slack = OUT_ATOL
        assert bool(((ob >= lo - slack) & (ob <= hi + slack)).all()), f"{name}: b={b} out of range"
