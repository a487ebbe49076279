"""Paged cache layout on the CPU: the oracle's gather restores the logical
cache the generator paged out, and paging changes no attention result."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from oracle_pins import make_case


def _gather_pin_holds(gather, page_size):
    """The pin: gathering the generator's pages (written apart from the
    oracle) gives back the logical cache on every valid token."""
    B, G, Tmax, D = 3, 2, 70, 8
    lens = np.array([70, 1, 33], dtype=np.int32)
    q, k, v, lens = make_case(B, 1, 4, G, D, Tmax, lens, seed=70)
    kp, vp, table = syn.paginate(k, v, lens, page_size, seed=71)
    kl = gather(kp, table, lens, table.shape[1] * page_size)
    return all(np.array_equal(kl[b, :, :int(lens[b])], k[b, :, :int(lens[b])]) for b in range(B))


@pytest.mark.parametrize("page_size", [8, 16, 64])
def test_gather_undoes_paginate(page_size):
    assert _gather_pin_holds(oracle.gather_pages, page_size)
    # physical pages are a permutation: no page serves two logical pages
    lens = [70, 1, 33]
    _, _, table = syn.paginate(np.zeros((3, 2, 70, 8), np.uint16), np.zeros((3, 2, 70, 8), np.uint16),
                               np.array(lens, np.int32), page_size, seed=71)
    used = [table[b, j] for b in range(3) for j in range(-(-lens[b] // page_size))]
    assert len(set(used)) == len(used)


def test_gather_pin_catches_planted_mistakes():
    """Copies of the gather with a plausible mistake fail the pin: the row
    within the page, the page index, and the KV-head axis."""
    def make(row_of, page_of, head_swap=False):
        def gather(k_pages, block_table, seq_lens, Tmax):
            num_pages, G, ps, D = k_pages.shape
            out = np.full((block_table.shape[0], G, Tmax, D), 0x7FC0, dtype=np.uint16)
            for b in range(block_table.shape[0]):
                for t in range(min(int(seq_lens[b]), Tmax)):
                    j = min(page_of(t, ps), block_table.shape[1] - 1)
                    page = k_pages[int(block_table[b, j])]
                    out[b, :, t, :] = (page[::-1] if head_swap else page)[:, row_of(t, ps) % ps, :]
            return out
        return gather

    assert _gather_pin_holds(make(lambda t, ps: t % ps, lambda t, ps: t // ps), 16)   # the right one
    assert not _gather_pin_holds(make(lambda t, ps: t // ps, lambda t, ps: t // ps), 16)
    assert not _gather_pin_holds(make(lambda t, ps: t % ps, lambda t, ps: t // ps + 1), 16)
    assert not _gather_pin_holds(make(lambda t, ps: t % ps, lambda t, ps: t // ps, head_swap=True), 16)


def test_paged_oracle_equals_contiguous_oracle():
    B, sq, H, G, D, Tmax = 2, 2, 8, 2, 16, 64
    q, k, v, lens = make_case(B, sq, H, G, D, Tmax, [64, 19], seed=72)
    kp, vp, table = syn.paginate(k, v, lens, 16, seed=73)
    a_out, a_lse = oracle.gqa_decode_paged_f64(q, kp, vp, table, lens, 0.25)
    b_out, b_lse = oracle.gqa_decode_f64(q, k, v, lens, 0.25)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)
