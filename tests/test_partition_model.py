"""A host-side model of the split-KV work partition (CPU only).

The split-KV kernel gives CTA c the tiles [c*W/P, (c+1)*W/P) of the flattened
(sequence, KV head, 64-token tile) list; a partial result goes to slot 0 if it
is the CTA's first segment, else slot 1; the CTA that merges unit u finds its
contributors as CTAs floor(((ub+1)P-1)/W) .. floor((ue*P-1)/W), skips CTAs with
an empty share and takes slot 0 when the CTA's share starts inside the unit.
This model restates those formulas and checks, over random ragged inputs, that
every tile is processed once, no slot is written twice, and the merge reads
exactly the slots that were written (and counts as many contributors as wrote
partials for the unit).
"""
import numpy as np
import pytest

TILE = 64


def tiles(lens, Tmax):
    t = np.clip(np.asarray(lens), 0, Tmax)
    return (t + TILE - 1) // TILE


def kernel_model(lens, G, Tmax, P):
    nt = tiles(lens, Tmax)
    pre = np.concatenate([[0], np.cumsum(nt * G)])
    W = int(pre[-1])
    written = {}          # (cta, slot) -> unit
    complete = set()
    covered = np.zeros(W, dtype=int)
    for c in range(P):
        lo, hi = c * W // P, (c + 1) * W // P
        x, b = lo, 0
        while x < hi:
            while x >= pre[b + 1]:
                b += 1
            g = (x - pre[b]) // nt[b]
            ub = pre[b] + g * nt[b]
            ue = ub + nt[b]
            e = min(hi, ue)
            covered[x:e] += 1
            if x == ub and e == ue:
                complete.add((b, g))
            else:
                slot = 0 if x == lo else 1
                assert (c, slot) not in written
                written[(c, slot)] = (b, g)
            x = e
    return W, pre, nt, written, complete, covered


def combine_model(b, g, pre, nt, W, P):
    if nt[b] == 0:
        return "empty", []
    ub = pre[b] + g * nt[b]
    ue = ub + nt[b]
    cf = ((ub + 1) * P - 1) // W
    cl = (ue * P - 1) // W
    if cf == cl:
        return "complete", []
    reads = []
    for c in range(cf, cl + 1):
        clo, chi = c * W // P, (c + 1) * W // P
        if clo >= chi:
            continue
        reads.append((c, 0 if clo >= ub else 1))
    return "split", reads


@pytest.mark.parametrize("seed", range(40))
def test_partition_and_combine_agree(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 12))
    G = int(rng.integers(1, 9))
    Tmax = int(rng.integers(1, 700))
    lens = rng.integers(-3, Tmax + 50, size=B)
    lens[rng.random(B) < 0.2] = 0
    P = int(rng.integers(1, 200))
    W, pre, nt, written, complete, covered = kernel_model(lens, G, Tmax, P)
    assert np.all(covered == 1)
    read = set()
    for b in range(B):
        for g in range(G):
            kind, reads = combine_model(b, g, pre, nt, W, P)
            if kind == "complete":
                assert (b, g) in complete
            elif kind == "split":
                assert (b, g) not in complete and len(reads) >= 2
                for r in reads:
                    assert written.get(r) == (b, g), (b, g, r)
                    read.add(r)
                assert len(reads) == sum(1 for u in written.values() if u == (b, g))
            else:
                assert nt[b] == 0
    assert read == set(written)   # every partial is merged, none is left over
