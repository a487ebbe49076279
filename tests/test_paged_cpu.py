"""Paged cache layout on the CPU: the oracle's gather restores the logical
cache the generator paged out, and paging changes no attention result."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle_pins import make_case


@pytest.mark.parametrize("page_size", [8, 16, 64])
def test_gather_undoes_paginate(page_size):
    B, G, Tmax, D = 3, 2, 70, 8
    lens = np.array([70, 1, 33], dtype=np.int32)
    q, k, v, lens = make_case(B, 1, 4, G, D, Tmax, lens, seed=70)
    kp, vp, table = syn.paginate(k, v, lens, page_size, seed=71)
    kl = oracle.gather_pages(kp, table, lens, table.shape[1] * page_size)
    for b in range(B):
        T = int(lens[b])
        assert np.array_equal(kl[b, :, :T], k[b, :, :T])
    # physical pages are a permutation: no page serves two logical pages
    used = [table[b, j] for b in range(B) for j in range(-(-int(lens[b]) // page_size))]
    assert len(set(used)) == len(used)


def test_paged_oracle_equals_contiguous_oracle():
    B, sq, H, G, D, Tmax = 2, 2, 8, 2, 16, 64
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [64, 19], seed=72)
    kp, vp, table = syn.paginate(k, v, lens, 16, seed=73)
    a_out, a_lse = oracle.gqa_decode_paged_f64(q, kp, vp, table, lens, 0.25)
    b_out, b_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.25)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)
