"""Pins of the oracle's lossless verification.

The pages give the rule: accept x_k with probability min(1, p(x_k)/q(x_k)), stop at the
first reject and draw the correction from norm(max(0, p - q)); the output then follows p
because min(q, p) + (p - min(p, q)) = p (billytse.dev DSpark page, section 1; xhh.club
page, Q&A on the acceptance rule).  The expected acceptance of one position equals
1 - 1/2 ||p - q||_1 (billytse.dev section 5.1; weigao.cc "3. confidence head").

Pins: Monte-Carlo acceptance against that closed form; chi-square tests that the emitted
tokens follow p (one position, and four positions with the scheduler in the loop); the
pages' look-ahead counterexample (golden fixture); and structural checks of the output.
"""
import json
import os

import numpy as np
from scipy import special, stats

import oracle
from workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rep(x, n):
    return np.broadcast_to(x, (n,) + x.shape).copy()


def _zeros_w(V, r=2):
    return np.zeros((V, r), np.uint16), np.zeros((r, V), np.uint16)


def test_single_position_acceptance_equals_one_minus_tv():
    V, n = 8, 200000
    rng = np.random.default_rng(0)
    U_row = rng.normal(size=(1, V)).astype(np.float32)
    T_rows = np.concatenate([U_row + rng.normal(size=(1, V)).astype(np.float32),
                             rng.normal(size=(1, V)).astype(np.float32)])
    W1, W2 = _zeros_w(V)
    U, T = _rep(U_row, n), _rep(T_rows, n)
    anchor = np.zeros(n, np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=1)
    v = oracle.verify(T, U, W1, W2, anchor, d["tokens"], np.ones(n, np.int32), seed=1)
    p = special.softmax(T_rows[0].astype(np.float64))
    q = special.softmax(U_row[0].astype(np.float64))
    want = 1.0 - 0.5 * np.abs(p - q).sum()
    assert abs(np.sum(np.minimum(p, q)) - want) < 1e-15       # the identity itself
    acc = v["accept_len"].mean()
    assert abs(acc - want) < 4.0 * np.sqrt(want * (1 - want) / n)
    # the emitted token (accepted draft or correction) follows p
    first = v["out_tokens"][:, 0]
    assert stats.chisquare(np.bincount(first, minlength=V), p * n).pvalue > 1e-3
    # when rejected, the correction lies where p > q
    rej = v["accept_len"] == 0
    assert np.all(p[first[rej]] > q[first[rej]])
    assert v["fallback"].sum() == 0


def test_four_positions_with_scheduler_in_the_loop_emit_target_distribution():
    # every request replicates the same U, T and Markov head; each gets its own random
    # stream.  Conditional on position k being emitted, its token follows softmax(T[k]).
    V, gamma, r, n = 8, 4, 4, 60000
    rng = np.random.default_rng(1)
    U_rows = rng.normal(size=(gamma, V)).astype(np.float32)
    T_rows = np.concatenate([U_rows + rng.normal(size=(gamma, V)).astype(np.float32),
                             rng.normal(size=(1, V)).astype(np.float32)])
    W1 = f32_to_bf16_bits(rng.normal(size=(V, r)).astype(np.float32))
    W2 = f32_to_bf16_bits(rng.normal(size=(r, V)).astype(np.float32))
    H = 4
    h = rng.normal(size=(n, gamma, H)).astype(np.float32)
    w_c = rng.normal(size=H + r).astype(np.float32)
    U, T = _rep(U_rows, n), _rep(T_rows, n)
    anchor = np.zeros(n, np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=2)
    _, a = oracle.confidence(h, anchor, d["tokens"], W1, w_c, 1.0)
    sps = (1.0 / (1.0 + 0.3 * np.arange(n * (gamma + 1) + 1) / n)).astype(np.float32)
    ell, _, _ = oracle.schedule(a.astype(np.float32), sps)
    assert 0 < ell.mean() < gamma
    v = oracle.verify(T, U, W1, W2, anchor, d["tokens"], ell, seed=2)
    for k in range(gamma + 1):
        emitted = v["n_out"] > k
        if emitted.sum() < 2000:
            continue
        p = special.softmax(T_rows[k].astype(np.float64))
        hist = np.bincount(v["out_tokens"][emitted, k], minlength=V)
        assert stats.chisquare(hist, p * emitted.sum()).pvalue > 1e-3, k


def test_lookahead_counterexample_matches_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "lookahead_counterexample.json")))
    V, n = 2, 400000
    p = np.array(g["target_p"])
    U_rows = np.zeros((1, V), np.float32)                   # q = (0.5, 0.5)
    T_rows = np.log(np.array([p, p])).astype(np.float32)    # row 1 and the bonus row
    W1, W2 = _zeros_w(V)
    U, T = _rep(U_rows, n), _rep(T_rows, n)
    anchor = np.zeros(n, np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=3)
    x1 = d["tokens"][:, 0]
    # non-anticipating: the verify length does not look at x_1
    v_na = oracle.verify(T, U, W1, W2, anchor, d["tokens"], np.ones(n, np.int32), seed=3)
    # look-ahead: verify position 1 only when c_2(x_1) is high, i.e. x_1 = A
    ell_la = (x1 == 0).astype(np.int32)
    v_la = oracle.verify(T, U, W1, W2, anchor, d["tokens"], ell_la, seed=3)
    for res, want in [(v_na, g["non_anticipating_output"]), (v_la, g["look_ahead_output"])]:
        freq_A = np.mean(res["out_tokens"][:, 0] == 0)
        assert abs(freq_A - want[0]) < 4.0 * np.sqrt(want[0] * want[1] / n), (freq_A, want)


def test_all_accepted_takes_the_bonus_from_row_l_plus_one():
    V, gamma, n = 16, 3, 32
    rng = np.random.default_rng(4)
    U_rows = rng.normal(size=(gamma, V)).astype(np.float32)
    bonus = np.full((1, V), -30.0, np.float32)
    bonus[0, 11] = 30.0
    T_rows = np.concatenate([U_rows, bonus])               # p = q on the draft rows
    W1, W2 = _zeros_w(V)
    U, T = _rep(U_rows, n), _rep(T_rows, n)
    anchor = np.zeros(n, np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=4)
    v = oracle.verify(T, U, W1, W2, anchor, d["tokens"], np.full(n, gamma, np.int32), seed=4)
    # p/q = 1 up to rounding: every test passes unless u sits in the rounding band
    assert np.all(v["accept_len"] == gamma)
    np.testing.assert_array_equal(v["out_tokens"][:, :gamma], d["tokens"])
    assert np.all(v["out_tokens"][:, gamma] == 11) and np.all(v["n_out"] == gamma + 1)


def test_zero_verified_length_is_plain_target_sampling_from_row_one():
    V, gamma, n = 8, 2, 60000
    rng = np.random.default_rng(5)
    U_rows = rng.normal(size=(gamma, V)).astype(np.float32)
    T_rows = rng.normal(size=(gamma + 1, V)).astype(np.float32)
    W1, W2 = _zeros_w(V)
    U, T = _rep(U_rows, n), _rep(T_rows, n)
    anchor = np.zeros(n, np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=6)
    v = oracle.verify(T, U, W1, W2, anchor, d["tokens"], np.zeros(n, np.int32), seed=6)
    assert np.all(v["accept_len"] == 0) and np.all(v["n_out"] == 1)
    assert np.all(v["out_tokens"][:, 1:] == -1)
    p = special.softmax(T_rows[0].astype(np.float64))
    assert stats.chisquare(np.bincount(v["out_tokens"][:, 0], minlength=V), p * n).pvalue > 1e-3


def test_output_structure():
    V, gamma, r, n = 50, 5, 4, 200
    rng = np.random.default_rng(7)
    U = rng.normal(size=(n, gamma, V)).astype(np.float32)
    T = np.concatenate([U + rng.normal(size=U.shape).astype(np.float32),
                        rng.normal(size=(n, 1, V)).astype(np.float32)], axis=1)
    W1 = f32_to_bf16_bits(rng.normal(size=(V, r)).astype(np.float32) * 0.1)
    W2 = f32_to_bf16_bits(rng.normal(size=(r, V)).astype(np.float32) * 0.1)
    anchor = rng.integers(0, V, n).astype(np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=7)
    ell = rng.integers(0, gamma + 1, n).astype(np.int32)
    v = oracle.verify(T, U, W1, W2, anchor, d["tokens"], ell, seed=7)
    assert np.all(v["accept_len"] <= ell) and np.all(v["n_out"] == v["accept_len"] + 1)
    for i in range(n):
        L = v["accept_len"][i]
        np.testing.assert_array_equal(v["out_tokens"][i, :L], d["tokens"][i, :L])
        assert 0 <= v["out_tokens"][i, L] < V
        assert np.all(v["out_tokens"][i, L + 1:] == -1)
        tested = ~np.isnan(v["band"][i])
        assert tested.sum() == min(ell[i], L + 1)
