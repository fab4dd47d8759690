"""Pins of the oracle's confidence head and survival product.

The pages define c_k = P(position k survives | positions < k accepted) produced by one
linear layer on [output_hidden_k ; markov_embedding(prev_token)] (weigao.cc DSpark-vs-MTP
page, "3. confidence head") and the survival a_j = prod_{i<=j} c_i (billytse.dev DSpark
page, section 5).  The Markov embedding is read as the W1 row of the predecessor.
"""
import numpy as np
from scipy import special

import oracle
from workloads import f32_to_bf16_bits

ONE_BF16 = 0x3F80


def test_zero_features_give_sigmoid_of_bias():
    n, gamma, H, V, r = 3, 5, 16, 32, 4
    h = np.zeros((n, gamma, H), np.float32)
    W1 = f32_to_bf16_bits(np.random.default_rng(0).normal(size=(V, r)).astype(np.float32))
    w_c = np.zeros(H + r, np.float32)
    c, a = oracle.confidence(h, np.zeros(n, np.int32), np.zeros((n, gamma), np.int32), W1, w_c, 1.0)
    c_exp = 1.0 / (1.0 + np.exp(-1.0))
    np.testing.assert_allclose(c, c_exp, rtol=1e-15)
    np.testing.assert_allclose(a, np.broadcast_to(c_exp ** np.arange(1, gamma + 1), a.shape), rtol=1e-14)


def test_hidden_part_one_hot_weight_matches_library_sigmoid():
    n, gamma, H, V, r = 4, 3, 8, 16, 2
    rng = np.random.default_rng(1)
    h = rng.normal(size=(n, gamma, H)).astype(np.float32)
    w_c = np.zeros(H + r, np.float32)
    w_c[5] = 1.0
    W1 = f32_to_bf16_bits(rng.normal(size=(V, r)).astype(np.float32))
    c, a = oracle.confidence(h, np.zeros(n, np.int32), np.zeros((n, gamma), np.int32), W1, w_c, -0.25)
    want = special.expit(h[:, :, 5].astype(np.float64) - 0.25)
    np.testing.assert_allclose(c, want, rtol=1e-14)
    np.testing.assert_allclose(a, np.cumprod(want, axis=1), rtol=1e-14)


def test_markov_part_uses_the_predecessor_row():
    # W1 rows one-hot on their own index and w_c[H + i] = s_i: the logit of position k is
    # s_{prev} + b_c with prev = anchor for k = 1 and the previous draft token after that
    n, gamma, H, V = 5, 4, 3, 6
    r = V
    W1 = np.zeros((V, r), np.uint16)
    W1[np.arange(V), np.arange(V)] = ONE_BF16
    s = np.array([-2.0, -1.0, 0.0, 0.5, 1.0, 3.0], np.float32)
    w_c = np.concatenate([np.zeros(H, np.float32), s])
    rng = np.random.default_rng(2)
    anchor = rng.integers(0, V, n).astype(np.int32)
    tokens = rng.integers(0, V, (n, gamma)).astype(np.int32)
    c, _ = oracle.confidence(np.zeros((n, gamma, H), np.float32), anchor, tokens, W1, w_c, 0.5)
    prev = np.concatenate([anchor[:, None], tokens[:, :-1]], axis=1)
    np.testing.assert_allclose(c, special.expit(s[prev].astype(np.float64) + 0.5), rtol=1e-14)


def test_survival_is_nonincreasing_and_starts_at_c1():
    n, gamma, H, V, r = 8, 16, 32, 64, 8
    rng = np.random.default_rng(3)
    h = rng.normal(size=(n, gamma, H)).astype(np.float32)
    W1 = f32_to_bf16_bits((rng.normal(size=(V, r)) * 0.5).astype(np.float32))
    w_c = (rng.normal(size=H + r) / np.sqrt(H + r)).astype(np.float32)
    c, a = oracle.confidence(h, rng.integers(0, V, n), rng.integers(0, V, (n, gamma)), W1, w_c, 1.0)
    assert np.all((c > 0) & (c < 1))
    np.testing.assert_array_equal(a[:, 0], c[:, 0])
    assert np.all(np.diff(a, axis=1) <= 0)
