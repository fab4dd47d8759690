"""Pins of the oracle's variants of the step: greedy drafting, verification of a greedy
draft, the asynchronous two-step capacity scheduler and fixed-threshold truncation.

Greedy drafting (billytse.dev DSpark page, section 11, where the serving example picks the
greedy draft sampling method) takes x_k = argmax_v z_v.  Its proposal is then the point
mass at x_k.  So the lossless rule of section 1 accepts x_k with probability p_k(x_k).
On a reject, the residual norm(max(0, p - q)) is p with x_k removed.  The pins reduce the
draft to numpy's argmax and scipy's softmax statistics.  They check a deterministic
transition chain.  They test by chi-square that the emitted tokens follow p.  They check
the closed-form acceptance p(x).

The two-step scheduler (weigao.cc DSpark-vs-MTP page, "4. hardware-aware prefix
scheduler"; billytse.dev section 7) fixes the count K from step t - 2 and takes the K
best positions of step t.  It is pinned by brute force: the first K items in the order of
a maximise the expected output among all prefix-feasible allocations of K positions.  It
is also pinned by the reduction to the synchronous scheduler when there is no history.

Fixed-threshold truncation (billytse.dev section 8; xhh.club page on load-dependent
thresholds) keeps the leading run of positions whose survival exceeds the threshold.  It
is pinned by counting with numpy on monotone a, and by hand cases of the strict and
first-failure rules.
"""
import itertools

import numpy as np
import pytest
from scipy import special, stats

import oracle
from workloads import f32_to_bf16_bits

ONE_BF16 = 0x3F80   # 1.0 in bf16


def _rep(x, n):
    return np.broadcast_to(x, (n,) + x.shape).copy()


# ------------------------------------------------------------------------ greedy draft

def test_greedy_draft_with_zero_weights_is_argmax_of_U():
    rng = np.random.default_rng(20)
    n, gamma, V = 6, 5, 300
    U = rng.normal(0, 3, size=(n, gamma, V)).astype(np.float32)
    W1 = f32_to_bf16_bits(rng.normal(size=(V, 16)).astype(np.float32))
    W2 = np.zeros((16, V), np.uint16)
    d = oracle.draft_greedy(U, W1, W2, rng.integers(0, V, n).astype(np.int32))
    np.testing.assert_array_equal(d["tokens"], U.argmax(-1))
    np.testing.assert_array_equal(d["q_tok"], 1.0)
    U64 = U.astype(np.float64)
    np.testing.assert_array_equal(d["row_max"], U64.max(-1))
    np.testing.assert_allclose(np.log(d["row_sumexp"]) + d["row_max"],
                               special.logsumexp(U64, axis=-1), rtol=1e-14)
    srt = np.sort(U64, axis=-1)
    np.testing.assert_array_equal(d["gap"], srt[..., -1] - srt[..., -2])


def test_greedy_draft_ties_go_to_the_smallest_index():
    V = 16
    U = np.zeros((1, 2, V), np.float32)
    U[0, 0, [3, 9, 12]] = 2.5
    U[0, 1, [7, 15]] = 1.0
    W1, W2 = np.zeros((V, 16), np.uint16), np.zeros((16, V), np.uint16)
    d = oracle.draft_greedy(U, W1, W2, np.zeros(1, np.int32))
    assert d["tokens"].tolist() == [[3, 7]]
    assert d["gap"].tolist() == [[0.0, 0.0]]


def test_greedy_draft_follows_the_transition_table():
    # W1[v] = e_{v mod r}, W2[i] = 20 * e_{next(i)}: the bias is +20 at next(prev), so the
    # greedy chain is anchor -> next(anchor) -> next(next(anchor)) ...
    V, r, gamma, n = 32, 16, 6, 4
    nxt = lambda v: (5 * v + 3) % r
    W1 = np.zeros((V, r), np.uint16)
    for v in range(V):
        W1[v, v % r] = ONE_BF16
    W2f = np.zeros((r, V), np.float32)
    for i in range(r):
        W2f[i, nxt(i)] = 20.0
    W2 = f32_to_bf16_bits(W2f)
    U = np.random.default_rng(21).normal(0, 1, size=(n, gamma, V)).astype(np.float32)
    anchor = np.array([0, 7, 19, 31], np.int32)
    d = oracle.draft_greedy(U, W1, W2, anchor)
    for b in range(n):
        prev, want = int(anchor[b]), []
        for _ in range(gamma):
            prev = nxt(prev % r)
            want.append(prev)
        assert d["tokens"][b].tolist() == want


# ---------------------------------------------------------------------- greedy verify

def test_greedy_single_position_accepts_with_probability_p_of_the_token():
    V, n = 8, 200000
    rng = np.random.default_rng(22)
    U_row = rng.normal(size=(1, V)).astype(np.float32)
    T_rows = np.concatenate([U_row + rng.normal(size=(1, V)).astype(np.float32),
                             rng.normal(size=(1, V)).astype(np.float32)])
    W1, W2 = np.zeros((V, 2), np.uint16), np.zeros((2, V), np.uint16)
    d = oracle.draft_greedy(_rep(U_row, n), W1, W2, np.zeros(n, np.int32))
    x = int(U_row[0].argmax())
    assert np.all(d["tokens"][:, 0] == x)
    v = oracle.verify_greedy(_rep(T_rows, n), d["tokens"], np.ones(n, np.int32), seed=5)
    p = special.softmax(T_rows[0].astype(np.float64))
    acc = v["accept_len"].mean()
    assert abs(acc - p[x]) < 4.0 * np.sqrt(p[x] * (1 - p[x]) / n)
    first = v["out_tokens"][:, 0]
    # the emitted token follows p; a correction is never the rejected token
    assert stats.chisquare(np.bincount(first, minlength=V), p * n).pvalue > 1e-3
    rej = v["accept_len"] == 0
    assert rej.sum() > 0 and np.all(first[rej] != x)
    # conditional on a reject, the correction follows p restricted to v != x
    pr = p.copy()
    pr[x] = 0.0
    pr /= pr.sum()
    hist = np.bincount(first[rej], minlength=V)
    keep = np.arange(V) != x
    assert stats.chisquare(hist[keep], (pr * rej.sum())[keep]).pvalue > 1e-3
    assert v["fallback"].sum() == 0


def test_greedy_draft_four_positions_threshold_truncated_emit_target_distribution():
    V, gamma, r, n = 8, 4, 4, 60000
    rng = np.random.default_rng(23)
    U = rng.normal(size=(n, gamma, V)).astype(np.float32)      # per-request drafts differ
    T_rows = rng.normal(size=(gamma + 1, V)).astype(np.float32)
    W1 = f32_to_bf16_bits(rng.normal(size=(V, r)).astype(np.float32))
    W2 = f32_to_bf16_bits(rng.normal(size=(r, V)).astype(np.float32))
    H = 4
    h = rng.normal(size=(n, gamma, H)).astype(np.float32)
    w_c = rng.normal(size=H + r).astype(np.float32)
    anchor = rng.integers(0, V, n).astype(np.int32)
    d = oracle.draft_greedy(U, W1, W2, anchor)
    _, a = oracle.confidence(h, anchor, d["tokens"], W1, w_c, 1.0)
    ell, _ = oracle.schedule_threshold(a.astype(np.float32), 0.3)
    assert 0 < ell.mean() < gamma
    v = oracle.verify_greedy(_rep(T_rows, n), d["tokens"], ell, seed=6)
    for k in range(gamma + 1):
        emitted = v["n_out"] > k
        if emitted.sum() < 2000:
            continue
        p = special.softmax(T_rows[k].astype(np.float64))
        hist = np.bincount(v["out_tokens"][emitted, k], minlength=V)
        assert stats.chisquare(hist, p * emitted.sum()).pvalue > 1e-3, k


def test_greedy_verify_equals_verify_of_a_point_mass_softmax_draft():
    # U rows with one logit 2000 above the rest: in fp64 softmax(U) is exactly the point
    # mass at the argmax, so the general verification must take the same decisions and
    # draw the same tokens as the greedy one on the same seed
    V, gamma, n = 64, 3, 300
    rng = np.random.default_rng(24)
    x = rng.integers(0, V, size=(n, gamma)).astype(np.int32)
    U = np.full((n, gamma, V), -1000.0, np.float32)
    np.put_along_axis(U, x[..., None], 1000.0, axis=-1)
    T = rng.normal(0, 1, size=(n, gamma + 1, V)).astype(np.float32)
    np.put_along_axis(T[:, :gamma], x[..., None], 1.5, axis=-1)
    W1, W2 = np.zeros((V, 16), np.uint16), np.zeros((16, V), np.uint16)
    anchor = np.zeros(n, np.int32)
    ell = rng.integers(0, gamma + 1, n).astype(np.int32)
    g = oracle.verify_greedy(T, x, ell, seed=7)
    s = oracle.verify(T, U, W1, W2, anchor, x, ell, seed=7)
    for key in ("accept_len", "out_tokens", "n_out", "fallback"):
        np.testing.assert_array_equal(g[key], s[key], err_msg=key)
    assert 0 < (g["accept_len"] < ell).sum() < n


# ------------------------------------------------------------------ async scheduler

def _best_k_allocation(a, K):
    """Brute force: the largest sum_r sum_{j<=l_r} a[r, j] over all l with sum l = K."""
    R, gamma = a.shape
    best = -1.0
    for ell in itertools.product(range(gamma + 1), repeat=R):
        if sum(ell) != K:
            continue
        best = max(best, sum(float(np.sum(a[r, :ell[r]].astype(np.float64))) for r in range(R)))
    return best


def test_async_without_history_equals_the_synchronous_scheduler():
    rng = np.random.default_rng(25)
    for R, gamma in [(1, 3), (3, 4), (7, 5), (40, 7)]:
        a = np.cumprod(rng.uniform(0.3, 1.0, size=(R, gamma)), axis=1).astype(np.float32)
        sps = (1.0 / (1.0 + 0.02 * np.arange(R * (gamma + 1) + 1))).astype(np.float32)
        ell, Bt, th = oracle.schedule(a, sps)
        ell2, Bt2, th2, K_out = oracle.schedule_async(a, sps, -1)
        np.testing.assert_array_equal(ell, ell2)
        assert Bt == Bt2 and th == th2 and K_out == Bt - R


@pytest.mark.parametrize("R,gamma", [(2, 3), (3, 3), (4, 2)])
def test_async_top_k_maximises_expected_output_for_its_capacity(R, gamma):
    rng = np.random.default_rng(26 + R)
    sps = (1.0 / (1.0 + 0.1 * np.arange(R * (gamma + 1) + 1))).astype(np.float32)
    for _ in range(10):
        a = np.cumprod(rng.uniform(0.05, 1.0, size=(R, gamma)), axis=1).astype(np.float32)
        for K in range(R * gamma + 1):
            ell, Bt, th, _ = oracle.schedule_async(a, sps, K)
            assert ell.sum() == K and Bt == R + K
            got = sum(float(np.sum(a[r, :ell[r]].astype(np.float64))) for r in range(R))
            assert abs(got - _best_k_allocation(a, K)) < 1e-6
            assert abs(th - (R + got) * float(sps[R + K])) < 1e-6 * (R + got)


def test_async_capacity_is_clamped_and_ties_break_by_request_then_position():
    a = np.array([[0.5, 0.5], [0.5, 0.25]], np.float32)
    sps = np.ones(7, np.float32)
    ell, Bt, _, _ = oracle.schedule_async(a, sps, 2)      # items (0,1) (0,2) (1,1) tie at 0.5
    assert ell.tolist() == [2, 0] and Bt == 4
    ell, Bt, _, _ = oracle.schedule_async(a, sps, 3)
    assert ell.tolist() == [2, 1]
    ell, Bt, _, _ = oracle.schedule_async(a, sps, 99)
    assert ell.tolist() == [2, 2] and Bt == 6


def test_async_pipeline_uses_the_capacity_of_two_steps_before():
    rng = np.random.default_rng(27)
    R, gamma, steps = 6, 5, 7
    sps = (1.0 / (1.0 + 0.05 * np.arange(R * (gamma + 1) + 1))).astype(np.float32)
    ring = [-1, -1]
    own = []
    for t in range(steps):
        # load varies from step to step, so the capacities differ
        a = np.cumprod(rng.uniform(0.2 + 0.1 * (t % 3), 1.0, size=(R, gamma)),
                       axis=1).astype(np.float32)
        ell, Bt, _, K_out = oracle.schedule_async(a, sps, ring[t % 2])
        own.append(oracle.schedule(a, sps)[1] - R)
        assert K_out == own[t]
        assert Bt - R == (own[t] if t < 2 else own[t - 2])
        ring[t % 2] = K_out
    assert len(set(own)) > 1


# ---------------------------------------------------------------- threshold truncation

def test_threshold_on_monotone_survival_counts_positions_above():
    rng = np.random.default_rng(28)
    a = np.cumprod(rng.uniform(0.3, 1.0, size=(50, 7)), axis=1).astype(np.float32)
    for th in [0.0, 0.1, 0.37, 0.6, 0.95, 1.0]:
        ell, Bt = oracle.schedule_threshold(a, th)
        want = np.sum(a > np.float32(th), axis=1)
        np.testing.assert_array_equal(ell, want)
        assert Bt == 50 + want.sum()


def test_threshold_is_strict_stops_at_the_first_failure_and_negative_keeps_all():
    a = np.array([[0.9, 0.3, 0.8], [0.5, 0.5, 0.5], [0.0, 0.0, 0.0]], np.float32)
    assert oracle.schedule_threshold(a, 0.5)[0].tolist() == [1, 0, 0]
    assert oracle.schedule_threshold(a, 0.25)[0].tolist() == [3, 3, 0]
    assert oracle.schedule_threshold(a, -1.0)[0].tolist() == [3, 3, 3]
    assert oracle.schedule_threshold(a, -1.0)[1] == 12
