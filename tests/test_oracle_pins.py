"""The oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    if pin.__name__ == "pin_bruteforce_mpmath":
        pytest.importorskip("mpmath")
    pin(oracle.get())


def test_row_range_and_threads_do_not_change_results():
    """Splitting rows over threads or computing them one range at a time gives
    the same bits as one sequential pass."""
    import numpy as np
    q, k, v, lens = oracle_pins.make_case(3, 2, 8, 2, 16, 40, [40, 13, 2], seed=30)
    full_o, full_l = oracle.get().gqa_decode(q, k, v, lens, 0.25)
    thr_o, thr_l = oracle.get().gqa_decode(q, k, v, lens, 0.25, threads=5)
    assert np.array_equal(full_o, thr_o) and np.array_equal(full_l, thr_l)
    part_o, part_l = oracle.get().gqa_decode(q, k, v, lens, 0.25, rows=(7, 19))
    flat_o = full_o.reshape(-1, 16)
    assert np.array_equal(part_o.reshape(-1, 16)[7:19], flat_o[7:19])
    assert np.all(np.isnan(part_o.reshape(-1, 16)[:7]))


def test_rejects_inputs_outside_the_definition():
    import numpy as np
    q, k, v, lens = oracle_pins.make_case(1, 1, 6, 4, 8, 5, [5], seed=31)  # 6 % 4 != 0
    with pytest.raises(ValueError):
        oracle.get().gqa_decode(q, k, v, lens, 0.3)
    q, k, v, lens = oracle_pins.make_case(1, 1, 4, 2, 8, 5, [5], seed=31)
    with pytest.raises(ValueError):
        oracle.get().gqa_decode(q, k, v, np.array([6], dtype=np.int32), 0.3)  # > Tmax


def test_wrong_axis_folds_are_caught():
    """Negative controls for the warning at the end of section 7 of the first
    page: folding the group into head_dim (summing different heads' dot
    products) or into the context axis (one softmax over all heads' keys)
    passes shape checks but changes the numbers; the comparison the pins use
    must tell them apart from the right fold."""
    import numpy as np
    q, k, v, lens = oracle_pins.make_case(1, 1, 8, 2, 16, 24, [24], seed=32)
    ref, _ = oracle_pins.sdpa_reference(q, k, v, lens)
    qf, kf, vf = (oracle_pins._f64(x) for x in (q, k, v))
    s = 0.25
    n_rep = 4
    wrong_d = np.zeros_like(ref)
    wrong_ctx = np.zeros_like(ref)
    for g in range(2):
        qg = qf[0, 0, g * n_rep:(g + 1) * n_rep]            # [4, D]
        # into head_dim: one score per key = sum over the group's heads
        x = s * (kf[0, g] @ qg.sum(axis=0))
        w = np.exp(x - x.max()); w /= w.sum()
        wrong_d[0, 0, g * n_rep:(g + 1) * n_rep] = w @ vf[0, g]
        # into ctx: one softmax over all (head, key) pairs of the group
        x = s * (qg @ kf[0, g].T)                          # [4, T]
        w = np.exp(x - x.max()); w /= w.sum()
        wrong_ctx[0, 0, g * n_rep:(g + 1) * n_rep] = w @ vf[0, g] * n_rep
    assert np.abs(wrong_d - ref).max() > 1e-2
    assert np.abs(wrong_ctx - ref).max() > 1e-2
