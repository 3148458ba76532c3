"""Pins for the worklist refinement steps of the oracle ("数据并行负载均衡"
§4.2 fitted load model, §4.4 phase 2 move/swap refinement after LPT)."""
import numpy as np
import pytest

import oracle
from packed_varlen_attention_cu_gb300 import workloads as W


def test_refine_hand_worked_move():
    # loads [27, 3]: moving the 10 leaves a gap of 4, swapping 10 for 1 leaves 6 -> move;
    # then the best candidates (move 9: 14, swap 9/1: 12) would not shrink the gap of 4
    a, loads, k = oracle.refine_move_swap([10, 9, 8, 1, 1, 1], [0, 0, 0, 1, 1, 1], 2, 20)
    assert a.tolist() == [1, 0, 0, 1, 1, 1] and loads.tolist() == [17, 13] and k == 1


def test_refine_hand_worked_swap():
    # loads [10, 5]: a move of 5 leaves a gap of 5 (no gain), a swap of 5 for 1 leaves 3
    a, loads, k = oracle.refine_move_swap([5, 5, 4, 1], [0, 0, 1, 1], 2, 20)
    assert a.tolist() == [1, 0, 1, 0] and loads.tolist() == [6, 9] and k == 1


def test_refine_stops_within_tolerance():
    # gap 4 of a largest load of 100 is under 5%: nothing moves
    a, loads, k = oracle.refine_move_swap([50, 50, 48, 48], [0, 0, 1, 1], 2, 20)
    assert k == 0 and a.tolist() == [0, 0, 1, 1]


def test_refine_invariants_random():
    rng = np.random.default_rng(11)
    for _ in range(200):
        n, bins = int(rng.integers(1, 40)), int(rng.integers(1, 6))
        cost = rng.integers(0, 1000, size=n)
        assign = rng.integers(0, bins, size=n)
        l0 = np.bincount(assign, weights=cost, minlength=bins).astype(np.int64)
        a, loads, k = oracle.refine_move_swap(cost, assign, bins, 20)
        assert 0 <= k <= 20
        assert np.array_equal(np.bincount(a, weights=cost, minlength=bins).astype(np.int64), loads)
        assert loads.sum() == l0.sum()
        if bins > 1:
            assert loads.max() - loads.min() <= l0.max() - l0.min()


def test_worklist_refinement_keeps_lpt_when_balanced():
    # LPT over ~100 units per bin is already within 5%: the refinement applies nothing
    w = W.tiny_pack()
    base = oracle.worklist(w.cu_seqlens, oracle.Mask(), 128, 128, 4, 4, num_ctas=7, c_tile=100)
    ref = oracle.worklist(w.cu_seqlens, oracle.Mask(), 128, 128, 4, 4, num_ctas=7, c_tile=100,
                          refine_iters=20)
    for key in ("units", "cta_off", "unit_cost"):
        np.testing.assert_array_equal(base[key], ref[key])


def test_fit_recovers_exact_model():
    rng = np.random.default_rng(2)
    P = rng.integers(10**6, 10**8, size=152)
    U = rng.integers(100, 5000, size=152)
    a, c = 0.002, 40.0
    t = a * P + c * U
    ct, coef = oracle.fit_tile_cost(P, U, t)
    assert ct == 20000
    np.testing.assert_allclose(coef, (a, c), rtol=1e-6)


def test_fit_matches_nnls_on_noisy_times():
    scipy_opt = pytest.importorskip("scipy.optimize")
    rng = np.random.default_rng(4)
    for trial in range(20):
        P = rng.integers(10**6, 10**8, size=152)
        U = rng.integers(100, 5000, size=152)
        # include cases whose unconstrained fit has a negative coefficient
        t = rng.uniform(-0.001, 0.003) * P + rng.uniform(-20, 60) * U + rng.normal(0, 2e4, 152)
        ct, coef = oracle.fit_tile_cost(P, U, t)
        X = np.stack([P, U], axis=1).astype(np.float64)
        ref, _ = scipy_opt.nnls(X, t)
        np.testing.assert_allclose(coef, ref, rtol=1e-6, atol=1e-9)
        if ref[0] > 0:
            assert ct == int(np.round(ref[1] / ref[0]))
        elif ref[1] > 0:
            assert ct == 1 << 24
        else:
            assert ct == -1


def test_fit_time_that_follows_tiles_alone():
    # pairs carry no time: the fit charges tiles only and returns the cap
    rng = np.random.default_rng(5)
    P = rng.integers(10**6, 10**8, size=152)
    U = rng.integers(100, 5000, size=152)
    ct, coef = oracle.fit_tile_cost(P, U, 30.0 * U - 1e-4 * P)
    assert ct == 1 << 24 and coef[0] == 0.0 and coef[1] > 0


def test_fit_degenerate():
    ct, _ = oracle.fit_tile_cost(np.zeros(8, dtype=np.int64), np.zeros(8, dtype=np.int64),
                                 np.ones(8))
    assert ct == -1
