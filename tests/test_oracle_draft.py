"""Pins of the oracle's draft (Markov bias + softmax + Gumbel-max).

The pages define p_k(v | x_<k) = softmax(U_k(v) + B_k(x_<k, v)) with the first-order
Markov bias B(x_{k-1}, .) = W1[x_{k-1}] W2 and a left-to-right loop that feeds each
sampled token back as the next predecessor (billytse.dev DSpark page, sections 3.2 and
3.3).  The pins below reduce the draft to library routines (scipy's softmax and
logsumexp) through special cases of W1 and W2, check the sampled frequencies against
the distribution with chi-square tests, and check the predecessor chaining with a
deterministic transition table.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle
from workloads import f32_to_bf16_bits

ONE_BF16 = 0x3F80   # 1.0 in bf16


def _replicated(row: np.ndarray, n: int) -> np.ndarray:
    return np.broadcast_to(row, (n,) + row.shape).copy()


def test_w_zero_is_plain_gumbel_max_on_U():
    V, n = 8, 60000
    U_row = np.array([[0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.9, 1.5]], dtype=np.float32)
    U = _replicated(U_row, n)
    W1 = np.zeros((V, 4), np.uint16)
    W2 = f32_to_bf16_bits(np.random.default_rng(1).normal(size=(4, V)).astype(np.float32))
    d = oracle.draft(U, W1, W2, np.zeros(n, np.int32), seed=11)
    p = special.softmax(U_row[0].astype(np.float64))
    hist = np.bincount(d["tokens"][:, 0], minlength=V)
    assert stats.chisquare(hist, p * n).pvalue > 1e-3
    # q_tok, row_max, row_sumexp against the library softmax / logsumexp
    x = d["tokens"][:, 0]
    np.testing.assert_allclose(d["q_tok"][:, 0], p[x], rtol=1e-13)
    np.testing.assert_allclose(d["row_max"][:, 0], U_row.max(), rtol=0)
    np.testing.assert_allclose(np.log(d["row_sumexp"][:, 0]) + d["row_max"][:, 0],
                               special.logsumexp(U_row[0].astype(np.float64)), rtol=1e-14)


def test_one_hot_W1_row_selects_W2_row():
    # W1[prev] = e_i makes the bias exactly the bf16 row W2[i]
    V, r, n = 8, 4, 50000
    rng = np.random.default_rng(2)
    U_row = rng.normal(size=(1, V)).astype(np.float32)
    W2f = rng.normal(size=(r, V)).astype(np.float32)
    W2 = f32_to_bf16_bits(W2f)
    W1 = np.zeros((V, r), np.uint16)
    prev, i = 5, 2
    W1[prev, i] = ONE_BF16
    d = oracle.draft(_replicated(U_row, n), W1, W2, np.full(n, prev, np.int32), seed=3)
    z = U_row[0].astype(np.float64) + (W2.astype(np.uint32) << 16).view(np.float32)[i].astype(np.float64)
    p = special.softmax(z)
    hist = np.bincount(d["tokens"][:, 0], minlength=V)
    assert stats.chisquare(hist, p * n).pvalue > 1e-3
    np.testing.assert_allclose(d["q_tok"][:, 0], p[d["tokens"][:, 0]], rtol=1e-13)
    np.testing.assert_allclose(np.log(d["row_sumexp"][0, 0]) + d["row_max"][0, 0],
                               special.logsumexp(z), rtol=1e-14)


def test_predecessor_chain_follows_transition_table():
    # W1 = identity rows, W2[t, succ(t)] = 40: the bias for prev t is +40 on succ(t) only,
    # so with small base logits every step must move to the successor of the previous token
    V, gamma, n = 8, 6, 64
    succ = np.array([3, 6, 0, 7, 1, 2, 5, 4])
    W1 = np.zeros((V, V), np.uint16)
    W1[np.arange(V), np.arange(V)] = ONE_BF16
    W2f = np.zeros((V, V), np.float32)
    W2f[np.arange(V), succ] = 40.0
    W2 = f32_to_bf16_bits(W2f)
    U = np.random.default_rng(4).normal(scale=0.5, size=(n, gamma, V)).astype(np.float32)
    anchor = np.arange(n, dtype=np.int32) % V
    d = oracle.draft(U, W1, W2, anchor, seed=5)
    prev = anchor.copy()
    for k in range(gamma):
        np.testing.assert_array_equal(d["tokens"][:, k], succ[prev])
        prev = d["tokens"][:, k]


def test_position_two_depends_on_sampled_position_one():
    # two-token toy from the pages' "of course" / "no problem" example: the Markov bias
    # couples position 2 to what position 1 actually sampled
    V, n = 4, 40000
    U = np.zeros((n, 2, V), np.float32)
    U[:, 0, 0] = U[:, 0, 1] = 3.0           # position 1: 'of' (0) or 'no' (1)
    U[:, 1, 2] = U[:, 1, 3] = 3.0           # position 2 marginal: 'course' (2) or 'problem' (3)
    W1 = np.zeros((V, V), np.uint16)
    W1[np.arange(V), np.arange(V)] = ONE_BF16
    W2f = np.zeros((V, V), np.float32)
    W2f[0, 2] = 6.0                         # after 'of' favour 'course'
    W2f[1, 3] = 6.0                         # after 'no' favour 'problem'
    d = oracle.draft(U, W1, f32_to_bf16_bits(W2f), np.full(n, 3, np.int32), seed=8)
    x1, x2 = d["tokens"][:, 0], d["tokens"][:, 1]
    mixed = np.mean(((x1 == 0) & (x2 == 3)) | ((x1 == 1) & (x2 == 2)))
    coherent = np.mean(((x1 == 0) & (x2 == 2)) | ((x1 == 1) & (x2 == 3)))
    assert coherent > 0.9 and mixed < 0.01


def test_equal_logits_sample_uniformly_and_ties_are_rare():
    V, n = 8, 40000
    U = np.zeros((n, 1, V), np.float32)
    d = oracle.draft(U, np.zeros((V, 2), np.uint16), np.zeros((2, V), np.uint16),
                     np.zeros(n, np.int32), seed=21)
    hist = np.bincount(d["tokens"][:, 0], minlength=V)
    assert stats.chisquare(hist).pvalue > 1e-3
    np.testing.assert_allclose(d["q_tok"], 1.0 / V, rtol=1e-14)
    assert np.all(d["gap"] > 0)


def test_seed_and_request_index_change_the_draws():
    V, n = 64, 16
    U = np.zeros((n, 3, V), np.float32)
    W1 = np.zeros((V, 2), np.uint16)
    W2 = np.zeros((2, V), np.uint16)
    a = oracle.draft(U, W1, W2, np.zeros(n, np.int32), seed=1)["tokens"]
    b = oracle.draft(U, W1, W2, np.zeros(n, np.int32), seed=2)["tokens"]
    c = oracle.draft(U, W1, W2, np.zeros(n, np.int32), seed=1, req_ids=np.arange(n) + 100)["tokens"]
    assert (a != b).mean() > 0.5 and (a != c).mean() > 0.5
    # the same (seed, request) reproduces the same path
    a2 = oracle.draft(U[3:4], W1, W2, np.zeros(1, np.int32), seed=1, req_ids=[3])["tokens"]
    np.testing.assert_array_equal(a2[0], a[3])
