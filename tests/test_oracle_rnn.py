"""Pins of the oracle's RNN head (weigao.cc DSpark-vs-MTP page, "2. Markov head and RNN
head").  One linear layer on [state ; previous-token embedding ; hidden state] gives the
gate, candidate and output blocks.  Then state_k = gate * state_{k-1} + (1 - gate) *
candidate and bias_k = W2 tanh(output).

The pins:
  * the hidden-state projection against numpy's matmul;
  * a saturated gate keeps the zero state exactly;
  * a closed gate makes the state the candidate (numpy);
  * constant gate and candidate give the exponential average (1 - lam^k) tanh(c0);
  * an output block on the token embedding makes the draft a transition chain (Gumbel-max
    recomputed with numpy from the pinned random draws);
  * an output block on the state carries the anchor into position 2 (closed form);
  * greedy tokens are the argmax of U + E W2;
  * verification with Markov rows equals the pinned Markov verification;
  * draft + verification emit the target distribution (chi-square).
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle
import workloads
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _rep(x, n):
    return np.broadcast_to(x, (n,) + x.shape).copy()


def _small(seed, n=4, gamma=4, V=64, r=16, H=8):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 1, size=(n, gamma, V)).astype(np.float32)
    h = rng.normal(0, 1, size=(n, gamma, H)).astype(np.float32)
    W1 = f32_to_bf16_bits(rng.normal(0, 0.5, size=(V, r)).astype(np.float32))
    W2 = f32_to_bf16_bits(rng.normal(0, 0.5, size=(r, V)).astype(np.float32))
    anchor = rng.integers(0, V, n).astype(np.int32)
    return rng, U, h, W1, W2, anchor


def test_projection_matches_numpy_matmul():
    rng = np.random.default_rng(50)
    n, H, r = 7, 40, 16
    h = rng.normal(size=(n, H)).astype(np.float32)
    W = f32_to_bf16_bits(rng.normal(size=(2 * r + H, 3 * r)).astype(np.float32))
    b = rng.normal(size=3 * r).astype(np.float32)
    hp = oracle.rnn_project(h, W, b)
    want = h.astype(np.float64) @ bf16_bits_to_f32(W)[2 * r:].astype(np.float64) + b
    np.testing.assert_allclose(hp, want, rtol=1e-12, atol=1e-12)


def test_saturated_gate_keeps_the_zero_state():
    rng, U, h, W1, W2, anchor = _small(51)
    r, H = 16, 8
    W = rng.normal(size=(2 * r + H, 3 * r)).astype(np.float32)
    W[:, :r] = 0.0                                   # gate weights
    b = rng.normal(size=3 * r).astype(np.float32)
    b[:r] = 60.0                                     # gate = 1 in double
    d = oracle.draft_rnn(U, h, W1, W2, f32_to_bf16_bits(W), b, anchor, seed=1)
    assert np.all(d["state"] == 0.0)


def test_closed_gate_makes_the_state_the_candidate():
    rng, U, h, W1, W2, anchor = _small(52)
    r, H, gamma = 16, 8, 4
    W = rng.normal(size=(2 * r + H, 3 * r)).astype(np.float32)
    W[:, :r] = 0.0
    W[:r, :] = 0.0                                   # no state input anywhere
    b = rng.normal(size=3 * r).astype(np.float32)
    b[:r] = -60.0                                    # gate ~ 1e-26
    Wb = f32_to_bf16_bits(W)
    d = oracle.draft_rnn(U, h, W1, W2, Wb, b, anchor, seed=2)
    Wf = bf16_bits_to_f32(Wb).astype(np.float64)
    prev = d["tokens"][:, gamma - 2]
    y_c = (bf16_bits_to_f32(W1)[prev].astype(np.float64) @ Wf[r:2 * r, r:2 * r]
           + h[:, gamma - 1].astype(np.float64) @ Wf[2 * r:, r:2 * r] + b[r:2 * r])
    np.testing.assert_allclose(d["state"], np.tanh(y_c), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("lam,c0", [(0.3, 0.8), (0.9, -1.7)])
def test_constant_gate_and_candidate_give_the_exponential_average(lam, c0):
    rng, U, h, W1, W2, anchor = _small(53)
    r, H, gamma = 16, 8, 4
    b = np.zeros(3 * r, np.float32)
    b[:r] = np.log(lam / (1 - lam))
    b[r:2 * r] = c0
    b[2 * r:] = 0.25
    d = oracle.draft_rnn(U, h, W1, W2, np.zeros((2 * r + H, 3 * r), np.uint16), b, anchor, seed=3)
    lam32 = 1.0 / (1.0 + np.exp(-np.float64(np.float32(np.log(lam / (1 - lam))))))
    want = (1.0 - lam32 ** gamma) * np.tanh(np.float64(np.float32(c0)))
    np.testing.assert_allclose(d["state"], want, rtol=1e-13)
    np.testing.assert_allclose(d["E"], np.tanh(0.25), rtol=1e-15)


def test_output_on_the_token_embedding_is_a_transition_chain():
    # output block = alpha * I on the embedding rows: E_k = tanh(alpha W1[x_{k-1}]); the
    # tokens must equal a numpy Gumbel-max over U_k + E_k W2 with the oracle's draws
    rng, U, h, W1, W2, anchor = _small(54)
    n, gamma, V, r, H, alpha, seed = 4, 4, 64, 16, 8, 1.5, 4
    W = np.zeros((2 * r + H, 3 * r), np.float32)
    W[r:2 * r, 2 * r:] = alpha * np.eye(r, dtype=np.float32)
    W[:, :2 * r] = rng.normal(size=(2 * r + H, 2 * r)).astype(np.float32)   # gate, candidate
    d = oracle.draft_rnn(U, h, W1, W2, f32_to_bf16_bits(W), rng.normal(size=3 * r).astype(np.float32) *
                         np.r_[np.ones(2 * r), np.zeros(r)].astype(np.float32), anchor, seed=seed)
    W1f = bf16_bits_to_f32(W1).astype(np.float64)
    W2f = bf16_bits_to_f32(W2).astype(np.float64)
    a32 = np.float64(np.float32(alpha))
    for b in range(n):
        prev = int(anchor[b])
        for k in range(1, gamma + 1):
            e = np.tanh(a32 * W1f[prev])
            z = U[b, k - 1].astype(np.float64) + e @ W2f
            g = np.array([oracle.gumbel(oracle.draw(seed, b, k, v, 0)) for v in range(V)])
            x = int(np.argmax(z + g))
            assert d["tokens"][b, k - 1] == x, (b, k)
            np.testing.assert_allclose(d["E"][b, k - 1], e, rtol=1e-14)
            prev = x


def test_output_on_the_state_carries_the_anchor_into_position_two():
    # output = alpha * state, candidate = beta * embedding, gate constant lam:
    # E_1 = tanh(0) = 0 (so x_1 is Gumbel-max on U_1 alone) and
    # E_2 = tanh(alpha (1 - lam) tanh(beta W1[anchor]))
    rng, U, h, W1, W2, anchor = _small(55)
    r, H, alpha, beta, lam, seed = 16, 8, 2.0, 0.75, 0.25, 5
    W = np.zeros((2 * r + H, 3 * r), np.float32)
    W[:r, 2 * r:] = alpha * np.eye(r, dtype=np.float32)
    W[r:2 * r, r:2 * r] = beta * np.eye(r, dtype=np.float32)
    b = np.zeros(3 * r, np.float32)
    b[:r] = np.log(lam / (1 - lam))
    d = oracle.draft_rnn(U, h, W1, W2, f32_to_bf16_bits(W), b, anchor, seed=seed)
    np.testing.assert_array_equal(d["E"][:, 0], 0.0)
    ref = oracle.draft(U[:, :1], W1, np.zeros_like(W2), anchor, seed=seed)
    np.testing.assert_array_equal(d["tokens"][:, 0], ref["tokens"][:, 0])
    lam32 = 1.0 / (1.0 + np.exp(-np.float64(b[0])))
    s1 = (1 - lam32) * np.tanh(0.75 * bf16_bits_to_f32(W1)[anchor].astype(np.float64))
    np.testing.assert_allclose(d["E"][:, 1], np.tanh(2.0 * s1), rtol=1e-13)


def test_greedy_tokens_are_the_argmax_of_the_projected_logits():
    rng, U, h, W1, W2, anchor = _small(56)
    w = workloads.scaled(workloads.get("tiny"), r=16, H=8)
    Wr, br = workloads.gen_rnn_weights(w)
    d = oracle.draft_rnn(U, h, W1, W2, Wr, br, anchor, seed=6, greedy=True)
    z = U.astype(np.float64) + np.einsum("bkr,rv->bkv", d["E"], bf16_bits_to_f32(W2).astype(np.float64))
    np.testing.assert_array_equal(d["tokens"], z.argmax(-1))
    np.testing.assert_array_equal(d["q_tok"], 1.0)


def test_verify_with_markov_rows_equals_the_markov_verification():
    rng = np.random.default_rng(57)
    n, gamma, V, r = 200, 3, 32, 16
    U = rng.normal(size=(n, gamma, V)).astype(np.float32)
    T = rng.normal(size=(n, gamma + 1, V)).astype(np.float32)
    W1 = f32_to_bf16_bits(rng.normal(0, 0.5, size=(V, r)).astype(np.float32))
    W2 = f32_to_bf16_bits(rng.normal(0, 0.5, size=(r, V)).astype(np.float32))
    anchor = rng.integers(0, V, n).astype(np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed=7)
    prev = np.concatenate([anchor[:, None], d["tokens"][:, :-1]], axis=1)
    E = bf16_bits_to_f32(W1)[prev].astype(np.float64)
    ell = rng.integers(0, gamma + 1, n).astype(np.int32)
    a = oracle.verify(T, U, W1, W2, anchor, d["tokens"], ell, seed=7)
    b = oracle.verify_rnn(T, U, E, W2, d["tokens"], ell, seed=7)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_rnn_draft_and_verification_emit_the_target_distribution():
    V, gamma, r, H, n = 8, 3, 16, 4, 60000
    rng = np.random.default_rng(58)
    U_rows = rng.normal(size=(gamma, V)).astype(np.float32)
    T_rows = rng.normal(size=(gamma + 1, V)).astype(np.float32)
    W1 = f32_to_bf16_bits(rng.normal(0, 0.5, size=(V, r)).astype(np.float32))
    W2 = f32_to_bf16_bits(rng.normal(0, 0.3, size=(r, V)).astype(np.float32))
    Wr = f32_to_bf16_bits(rng.normal(0, 0.5, size=(2 * r + H, 3 * r)).astype(np.float32))
    br = rng.normal(0, 0.5, size=3 * r).astype(np.float32)
    h = rng.normal(size=(n, gamma, H)).astype(np.float32)
    anchor = rng.integers(0, V, n).astype(np.int32)
    d = oracle.draft_rnn(_rep(U_rows, n), h, W1, W2, Wr, br, anchor, seed=8)
    v = oracle.verify_rnn(_rep(T_rows, n), _rep(U_rows, n), d["E"], W2, d["tokens"],
                          np.full(n, gamma, np.int32), seed=8)
    assert 0.1 < v["accept_len"].mean() < gamma - 0.1
    for k in range(gamma + 1):
        emitted = v["n_out"] > k
        if emitted.sum() < 2000:
            continue
        p = special.softmax(T_rows[k].astype(np.float64))
        hist = np.bincount(v["out_tokens"][emitted, k], minlength=V)
        assert stats.chisquare(hist, p * emitted.sum()).pvalue > 1e-3, k
