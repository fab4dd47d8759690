"""Pins of the oracle's hardware-aware prefix scheduler.

The pages define B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r} a_{r,j}) and the goal
max Theta = tau * SPS(B); positions are added in descending order of expected return and
the scheduler stops as soon as Theta would fall (billytse.dev DSpark page, section 6;
early stopping, section 7).  The xhh.club page states the equivalent marginal rule: add a
position while its survival exceeds the expected output times the slow-down ratio.

Pins: brute force over every (l_1..l_R) on tiny batches (greedy = global optimum when
f(n) = (R + S_n) SPS(R + n) is quasi-concave), the marginal rule at every admission and
at the stop, a hand-worked example, early stopping on a jagged table, and load
monotonicity.
"""
import itertools

import numpy as np

import oracle


def _theta(a, ell, sps):
    R = a.shape[0]
    tau = R + sum(float(np.sum(a[r, :ell[r]].astype(np.float64))) for r in range(R))
    return tau * float(sps[R + int(np.sum(ell))])


def _random_a(rng, R, gamma):
    c = rng.uniform(0.05, 1.0, size=(R, gamma))
    return np.cumprod(c, axis=1).astype(np.float32)


def test_hand_worked_example():
    a = np.array([[0.9, 0.5], [0.8, 0.1]], np.float32)
    sps = np.array([1, 1, 1, 1, 0.8, 0.5, 0.4], np.float32)
    # Theta: start 2*1=2; +0.9 -> 2.9*SPS(3)=2.9; +0.8 -> 3.7*SPS(4)=2.96; +0.5 -> 4.2*0.5=2.1 stop
    ell, Bt, th = oracle.schedule(a, sps)
    assert ell.tolist() == [1, 1] and Bt == 4
    assert abs(th - float(np.float32(0.9) + np.float32(0.8) + 2) * float(np.float32(0.8))) < 1e-6


def test_greedy_is_global_optimum_for_concave_curve():
    rng = np.random.default_rng(0)
    for trial in range(60):
        R, gamma = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        a = _random_a(rng, R, gamma)
        sps = (1.0 / (1.0 + 0.01 * np.arange(R * (gamma + 1) + 1) * rng.uniform(1, 30))).astype(np.float32)
        ell, Bt, th = oracle.schedule(a, sps)
        best = max(_theta(a, e, sps) for e in itertools.product(range(gamma + 1), repeat=R))
        assert abs(th - best) <= 1e-9 * best, (trial, a, ell)
        assert Bt == R + int(ell.sum())
        assert abs(_theta(a, ell, sps) - th) <= 1e-9 * th


def test_marginal_rule_holds_at_every_admission_and_fails_at_the_stop():
    rng = np.random.default_rng(1)
    for _ in range(40):
        R, gamma = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        a = _random_a(rng, R, gamma)
        sps = (1.0 / (1.0 + 0.02 * np.maximum(0, np.arange(R * (gamma + 1) + 1) - rng.integers(0, 2 * R)))
               ).astype(np.float32)
        ell, Bt, _ = oracle.schedule(a, sps)
        # every admitted item beats tau * (SPS(B)/SPS(B+1) - 1) at its admission, in sorted order
        items = sorted(((float(a[r, j]), r, j) for r in range(R) for j in range(gamma)),
                       key=lambda t: (-t[0], t[1], t[2]))
        tau, B = float(R), R
        admitted = int(ell.sum())
        for n, (av, r, j) in enumerate(items):
            thresh = tau * (float(sps[B]) / float(sps[B + 1]) - 1.0)
            if n < admitted:
                assert av > thresh - 1e-9
                tau += av
                B += 1
            else:
                assert av <= thresh + 1e-9
                break
        # admitted sets are prefixes of each request's block
        for r in range(R):
            assert 0 <= ell[r] <= gamma


def test_first_non_rise_stops_even_if_a_later_point_is_higher():
    # a jagged curve: a dip at B = R + 2 and a rise after it; early stopping halts at the
    # dip although admitting more would give a larger Theta later (non-anticipating rule)
    R, gamma = 1, 4
    a = np.array([[0.95, 0.9, 0.85, 0.8]], np.float32)
    sps = np.array([1.0, 1.0, 1.0, 0.5, 0.9, 0.9], np.float32)
    ell, Bt, th = oracle.schedule(a, sps)
    assert ell.tolist() == [1] and Bt == 2
    assert _theta(a, [4], sps) > th


def test_lighter_load_verifies_more():
    rng = np.random.default_rng(2)
    R, gamma = 16, 8
    a = _random_a(rng, R, gamma)
    n = np.arange(R * (gamma + 1) + 1)
    totals = []
    for slope in [0.0005, 0.002, 0.01, 0.05]:
        ell, _, _ = oracle.schedule(a, (1.0 / (1.0 + slope * n)).astype(np.float32))
        totals.append(int(ell.sum()))
    assert totals == sorted(totals, reverse=True) and totals[0] > totals[-1]


def test_flat_curve_admits_everything_with_positive_survival():
    a = np.array([[0.5, 0.25], [0.0, 0.0]], np.float32)
    sps = np.ones(2 * 3 + 1, np.float32)
    ell, Bt, _ = oracle.schedule(a, sps)
    assert ell.tolist() == [2, 0] and Bt == 4


def test_ties_are_broken_by_request_then_position():
    a = np.array([[0.5, 0.5], [0.5, 0.5]], np.float32)
    sps = np.array([1.0, 1.0, 1.0, 1.0, 0.7, 0.5, 0.4], np.float32)
    # 2 -> 2.5 (B=3) -> 3.0*0.7=2.1 stops: the single admitted tie goes to request 0
    ell, Bt, _ = oracle.schedule(a, sps)
    assert ell.tolist() == [1, 0] and Bt == 3
