"""Parity of the CUDA path with the oracle on the degenerate and extreme shapes.

The shapes cover: one request and one position; the smallest vocabulary (8, one ragged
128-row tile, a grid of one CTA); the largest block (gamma = 32, every lane of the
decision warp); a second request chunk holding a single request; a rank that is not a
multiple of 32 (r = 48, 16-row K chunks); a vocabulary of exactly one tile.  They also
cover the acceptance extremes: every position accepted (target = draft distribution,
bonus from the last row) and every first position rejected (a target peaked elsewhere),
and a residual whose every logit is a race candidate.
The tie band and tolerances are those of the main parity tests.
"""
import numpy as np
import pytest

import oracle
import workloads
from _parity import verify_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
ds = pytest.importorskip("speculative_decoding_03_gb300")

TIE = 1e-5
RTOL = 1e-5

BASE = workloads.get("qwen3_4b_like")
SHAPES = {
    "B1_g1_V8": workloads.scaled(BASE, B=1, gamma=1, V=8, r=16, H=4),
    "B1_g32": workloads.scaled(BASE, B=1, gamma=32, V=264, r=16, H=4),
    "B2_g32_r48": workloads.scaled(BASE, B=2, gamma=32, V=392, r=48, H=8),
    "B17_r48": workloads.scaled(BASE, B=17, gamma=2, V=136, r=48, H=8),
    "B33_V128": workloads.scaled(BASE, B=33, gamma=3, V=128, r=32, H=4),
}


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _first_divergence_ok(got, ref, gap):
    """Tokens equal until the first tie-band position of each row."""
    for i in range(got.shape[0]):
        for k in range(got.shape[1]):
            if got[i, k] != ref[i, k]:
                assert gap[i, k] <= TIE, (i, k, got[i, k], ref[i, k], gap[i, k])
                return False
    return True


@pytest.mark.parametrize("name", list(SHAPES))
def test_step_on_edge_shapes(name):
    _need_gpu()
    w = SHAPES[name]
    inp = workloads.generate(w)
    step = ds.Step(ds.to_device(inp), float(inp.b_c)).run(seed=w.seed)
    got = step.results()
    ref = oracle.step(inp, seed=w.seed)
    assert step.ws.status() == 0
    if not _first_divergence_ok(got["tokens"], ref["draft"]["tokens"], ref["draft"]["gap"]):
        return
    for key in ("q_tok", "row_max", "row_sumexp"):
        np.testing.assert_allclose(got[key], ref["draft"][key], rtol=RTOL, err_msg=key)
    np.testing.assert_allclose(got["c"], ref["c"], rtol=RTOL)
    np.testing.assert_allclose(got["a"], ref["a"], rtol=RTOL)
    # the oracle's chain schedules its own survivals: the same l unless a stop decision sits
    # within the two chains' rounding, which seeded data does not produce
    np.testing.assert_array_equal(got["ell"], ref["ell"])
    assert got["B_total"] == ref["B_total"]
    verify_rows(got, ref["verify"], name)
    np.testing.assert_array_equal(got["n_out"], got["accept_len"] + 1)


def _manual(B, gamma, V, r, seed):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2, size=(B, gamma, V)).astype(np.float32)
    W1 = np.zeros((V, r), np.uint16)                       # no Markov bias: z = U exactly
    W2 = workloads.f32_to_bf16_bits(rng.normal(0, 0.02, size=(r, V)).astype(np.float32))
    anchor = rng.integers(0, V, B).astype(np.int32)
    return rng, U, W1, W2, anchor


def _run(U, T, W1, W2, anchor, ell, seed):
    B, gamma, V = U.shape
    r = W1.shape[1]
    ws = ds.Workspace(B, gamma, V, r)
    cu = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x, dtype=dt)).cuda()
    W1d, W2d = ds.as_bf16_tensor(W1), ds.as_bf16_tensor(W2)
    d = ds.draft(cu(U, np.float32), W1d, W2d, cu(anchor, np.int32), seed, ws)
    out = ds.verify(cu(T, np.float32), cu(U, np.float32), W1d, W2d, cu(anchor, np.int32), d["tokens"],
                    d["q_tok"], d["row_max"], d["row_sumexp"], cu(ell, np.int32), seed, ws)
    assert ws.status() == 0
    return {k: v.cpu().numpy() for k, v in d.items()}, {k: v.cpu().numpy() for k, v in out.items()}


def test_target_equal_to_draft_accepts_every_position_and_takes_the_bonus():
    _need_gpu()
    B, gamma, V, r, seed = 64, 6, 1000, 16, 21
    rng, U, W1, W2, anchor = _manual(B, gamma, V, r, seed)
    T = np.concatenate([U, rng.normal(0, 2, size=(B, 1, V)).astype(np.float32)], axis=1)
    ell = np.full(B, gamma, np.int32)
    d, v = _run(U, T, W1, W2, anchor, ell, seed)
    ref_d = oracle.draft(U, W1, W2, anchor, seed)
    if not _first_divergence_ok(d["tokens"], ref_d["tokens"], ref_d["gap"]):
        pytest.skip("a draft decision in the tie band (the verification then sees other tokens)")
    ref = oracle.verify(T, U, W1, W2, anchor, ref_d["tokens"], ell, seed)
    # p = q at every position: everything is accepted except inside the band |u - 1| <= 1e-5
    np.testing.assert_array_equal(ref["accept_len"], gamma)
    inside = np.nanmin(ref["band"], axis=1) <= TIE
    assert np.all(v["accept_len"][~inside] == gamma)
    np.testing.assert_array_equal(v["out_tokens"][~inside, :gamma], d["tokens"][~inside])
    same = ~inside & (ref["gap"] > TIE)
    np.testing.assert_array_equal(v["out_tokens"][same, gamma], ref["out_tokens"][same, gamma])


def test_target_peaked_elsewhere_rejects_every_first_position():
    _need_gpu()
    B, gamma, V, r, seed = 64, 4, 1000, 16, 22
    rng, U, W1, W2, anchor = _manual(B, gamma, V, r, seed)
    d0 = oracle.draft(U, W1, W2, anchor, seed)
    T = rng.normal(0, 1, size=(B, gamma + 1, V)).astype(np.float32)
    peak = (d0["tokens"][:, 0] + 1 + rng.integers(0, V - 1, B)) % V
    T[np.arange(B), 0, peak] = 40.0                       # p(x_1) ~ e^-40
    ell = np.full(B, gamma, np.int32)
    d, v = _run(U, T, W1, W2, anchor, ell, seed)
    np.testing.assert_array_equal(d["tokens"][:, 0], d0["tokens"][:, 0])
    np.testing.assert_array_equal(v["accept_len"], 0)
    np.testing.assert_array_equal(v["n_out"], 1)
    np.testing.assert_array_equal(v["out_tokens"][:, 0], peak)       # the residual's mass
    np.testing.assert_array_equal(v["out_tokens"][:, 1:], -1)


def test_residual_whose_every_logit_is_a_race_candidate():
    """A residual with P barely above Q on every logit: the target row is the draft's own
    logits except the drafted token, 30 lower, so position 1 is rejected and P - Q is about
    q(x_1) Q everywhere else, below the race's error allowance: no lower bound survives and
    every logit of a segment is a candidate (more than a segment's candidate list holds, so
    the segments score them themselves).  The draw matches the oracle wherever the oracle's
    top-two gap is above the fp32 rounding of log(P - Q) (about 1e-2 here)."""
    _need_gpu()
    B, gamma, V, r, seed = 16, 2, 8192, 16, 23
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 0.1, size=(B, gamma, V)).astype(np.float32)     # q(x) ~ 1 / V
    W1 = np.zeros((V, r), np.uint16)                                  # z = U exactly
    W2 = workloads.f32_to_bf16_bits(rng.normal(0, 0.02, size=(r, V)).astype(np.float32))
    anchor = rng.integers(0, V, B).astype(np.int32)
    d0 = oracle.draft(U, W1, W2, anchor, seed)
    T = np.concatenate([U, rng.normal(0, 1, size=(B, 1, V)).astype(np.float32)], axis=1)
    T[np.arange(B), 0, d0["tokens"][:, 0]] -= 30.0
    ell = np.full(B, gamma, np.int32)
    d, v = _run(U, T, W1, W2, anchor, ell, seed)
    np.testing.assert_array_equal(d["tokens"][:, 0], d0["tokens"][:, 0])
    np.testing.assert_array_equal(v["accept_len"], 0)
    np.testing.assert_array_equal(v["n_out"], 1)
    assert np.all(v["out_tokens"][:, 0] != d0["tokens"][:, 0])      # outside the residual
    assert np.all((v["out_tokens"][:, 0] >= 0) & (v["out_tokens"][:, 0] < V))
    ref = oracle.verify(T, U, W1, W2, anchor, d0["tokens"], ell, seed)
    np.testing.assert_array_equal(ref["accept_len"], 0)
    clear = ref["gap"] > 5e-2
    assert clear.sum() >= B // 2
    np.testing.assert_array_equal(v["out_tokens"][clear, 0], ref["out_tokens"][clear, 0])


def test_verify_with_more_rows_than_a_grid_dimension():
    """B * gamma = 65536 verified rows (one more than a grid's y extent): the statistics
    kernel folds them and the outcomes match the oracle."""
    _need_gpu()
    B, gamma, V, r, seed = 4096, 16, 64, 16, 31
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2, size=(B, gamma, V)).astype(np.float32)
    T = (np.concatenate([U, rng.normal(0, 2, size=(B, 1, V)).astype(np.float32)], axis=1) +
         rng.normal(0, 1, size=(B, gamma + 1, V)).astype(np.float32))
    W1 = workloads.f32_to_bf16_bits(rng.normal(0, 0.02, size=(V, r)).astype(np.float32))
    W2 = workloads.f32_to_bf16_bits(rng.normal(0, 0.02, size=(r, V)).astype(np.float32))
    anchor = rng.integers(0, V, B).astype(np.int32)
    ell = np.full(B, gamma, np.int32)
    d = oracle.draft(U, W1, W2, anchor, seed)
    ref = oracle.verify(T, U, W1, W2, anchor, d["tokens"], ell, seed)
    ws = ds.Workspace(B, gamma, V, r)
    cu = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x, dtype=dt)).cuda()
    out = ds.verify(cu(T, np.float32), cu(U, np.float32), ds.as_bf16_tensor(W1), ds.as_bf16_tensor(W2),
                    cu(anchor, np.int32), cu(d["tokens"], np.int32), cu(d["q_tok"], np.float32),
                    cu(d["row_max"], np.float32), cu(d["row_sumexp"], np.float32), cu(ell, np.int32),
                    seed, ws)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert ws.status() == 0
    verify_rows(got, ref, "B4096_g16")
    assert np.mean(got["accept_len"] == ref["accept_len"]) > 0.999
