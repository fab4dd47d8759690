"""Pins of the oracle's Markov transition bias alone (``oracle.markov_bias``).

billytse.dev DSpark page, section 3.3: the first-order Markov head adds
B(x_{k-1}, .) = W1[x_{k-1}] W2 (rank r) to the base logits; W1 is the previous token's
small embedding [V, r] and W2 projects it back to the vocabulary [r, V].  The oracle
forms each row with a plain double loop over the rank.  What pins it here, none of which
goes through that loop:
  * a one-hot W1 row makes the bias exactly one bf16 row of W2 (bit for bit);
  * two-hot rows with power-of-two coefficients give an exact linear combination of two
    W2 rows;
  * a rank-one W2 = alpha beta^T gives the closed form (W1[prev] . alpha) beta;
  * brute force over every (i, v) of a tiny case, term by term in Python floats;
  * numpy's fp64 matmul on random bf16 weights with r != V (a transposed W2 index or a
    dropped rank term fails it);
  * a predecessor of -1 is a zero row, and other out-of-range ids are rejected.
"""
import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _bf16_scalar(x):
    return _bf16([x])[0]


def test_one_hot_row_is_a_w2_row_bit_for_bit():
    V, r = 40, 12
    rng = np.random.default_rng(1)
    W2 = _bf16(rng.normal(size=(r, V)))
    W1 = np.zeros((V, r), np.uint16)
    for t in range(V):
        W1[t, t % r] = 0x3F80                       # 1.0
    prev = np.array([0, 5, 13, 39, 11], np.int32)
    got = oracle.markov_bias(W1, W2, prev)
    want = bf16_bits_to_f32(W2)[prev % r].astype(np.float64)
    np.testing.assert_array_equal(got, want)


def test_two_hot_rows_give_exact_linear_combinations():
    V, r = 24, 6
    rng = np.random.default_rng(2)
    W2 = _bf16(rng.normal(size=(r, V)))
    W2f = bf16_bits_to_f32(W2).astype(np.float64)
    W1 = np.zeros((V, r), np.uint16)
    W1[3, 1], W1[3, 4] = _bf16_scalar(0.5), _bf16_scalar(-2.0)
    W1[7, 0], W1[7, 5] = _bf16_scalar(0.25), _bf16_scalar(4.0)
    got = oracle.markov_bias(W1, W2, np.array([3, 7], np.int32))
    np.testing.assert_array_equal(got[0], 0.5 * W2f[1] - 2.0 * W2f[4])
    np.testing.assert_array_equal(got[1], 0.25 * W2f[0] + 4.0 * W2f[5])


def test_rank_one_projection_closed_form():
    # W2[i, v] = alpha_i beta_v with powers of two (exact in bf16 and in every product)
    V, r = 32, 8
    rng = np.random.default_rng(3)
    alpha = 2.0 ** rng.integers(-3, 3, size=r) * rng.choice([-1, 1], size=r)
    beta = 2.0 ** rng.integers(-4, 2, size=V) * rng.choice([-1, 1], size=V)
    W2 = _bf16(np.outer(alpha, beta))
    W1f = np.round(rng.normal(size=(V, r)) * 8) / 8          # few bits: exact in bf16
    W1 = _bf16(W1f)
    prev = rng.integers(0, V, size=10).astype(np.int32)
    got = oracle.markov_bias(W1, W2, prev)
    want = np.outer(W1f[prev] @ alpha, beta)
    np.testing.assert_array_equal(got, want)


def test_brute_force_term_by_term():
    V, r = 8, 4
    rng = np.random.default_rng(4)
    W1 = _bf16(rng.normal(size=(V, r)))
    W2 = _bf16(rng.normal(size=(r, V)))
    prev = np.array([6, 0, 3], np.int32)
    got = oracle.markov_bias(W1, W2, prev)
    w1 = bf16_bits_to_f32(W1).tolist()
    w2 = bf16_bits_to_f32(W2).tolist()
    for n, t in enumerate(prev.tolist()):
        for v in range(V):
            s = 0.0
            for i in range(r):
                s += float(w1[t][i]) * float(w2[i][v])
            assert got[n, v] == pytest.approx(s, rel=1e-15, abs=1e-300)


def test_random_weights_against_numpy_matmul():
    V, r = 301, 48                  # r != V: a transposed W2 index reads the wrong entries
    rng = np.random.default_rng(5)
    W1 = _bf16(rng.normal(scale=0.02, size=(V, r)))
    W2 = _bf16(rng.normal(scale=0.02, size=(r, V)))
    prev = rng.integers(0, V, size=17).astype(np.int32)
    got = oracle.markov_bias(W1, W2, prev)
    want = bf16_bits_to_f32(W1).astype(np.float64)[prev] @ bf16_bits_to_f32(W2).astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-18)
    # each rank term matters: dropping any one changes the rows
    for i in (0, r // 2, r - 1):
        W2d = W2.copy()
        W2d[i] = 0
        assert np.max(np.abs(oracle.markov_bias(W1, W2d, prev) - got)) > 1e-6


def test_missing_predecessor_is_a_zero_row_and_bad_ids_are_rejected():
    V, r = 16, 4
    rng = np.random.default_rng(6)
    W1 = _bf16(rng.normal(size=(V, r)))
    W2 = _bf16(rng.normal(size=(r, V)))
    got = oracle.markov_bias(W1, W2, np.array([-1, 2, -1], np.int32))
    assert np.all(got[0] == 0) and np.all(got[2] == 0) and np.any(got[1] != 0)
    for bad in (V, -2):
        with pytest.raises(ValueError):
            oracle.markov_bias(W1, W2, np.array([bad], np.int32))
