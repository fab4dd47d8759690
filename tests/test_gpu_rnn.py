"""Parity of the CUDA RNN head with the CPU oracle: the weight packing, the hidden-state
projection, the RNN draft (Gumbel and greedy), its verification and the whole step.

The bars match the main parity tests.  Tokens must be bit-exact except inside the tie
band (top-two score gap within 1e-5, or |u - p/q| within 1e-5).  q_tok, row max and sum
must be within 1e-5 relative.  The head's output rows E and the projection must be within
1e-5 of the oracle's fp64 values, scaled by the magnitude of the terms summed.  Each call
is fed the oracle's upstream outputs: the projection, and the draft's tokens and rows.
"""
import numpy as np
import pytest

import oracle
import workloads
from _parity import assert_rate, band_cases_draft, band_cases_verify, draft_rows, verify_rows
from workloads import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
ds = pytest.importorskip("speculative_decoding_03_gb300")

TIE = 1e-5
RTOL = 1e-5

CASES = {
    "tiny": workloads.get("tiny"),
    "qwen_small": workloads.scaled(workloads.get("qwen3_4b_like"), B=5, gamma=3, V=904, r=64, H=32),
    "prod_small": workloads.scaled(workloads.get("production"), B=40, gamma=5, V=2056, r=256, H=64),
    "long_small": workloads.scaled(workloads.get("long_block"), B=7, gamma=15, V=1032, r=256, H=16,
                                   noise_std=lambda k: 0.5 + 1.5 * (k - 1) / 14.0),
    "wide_batch": workloads.scaled(workloads.get("scheduler_stress"), B=300, gamma=2, V=520, r=128, H=8),
}


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _cuda(x, dt):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=dt)).cuda()


def _setup(w, with_T=True, requests=None):
    inp = workloads.generate(w, requests=requests, with_T=with_T)
    W_rnn, b_rnn = workloads.gen_rnn_weights(w)
    dev = ds.rnn_to_device(W_rnn, b_rnn, ds.to_device(inp))
    return inp, W_rnn, b_rnn, dev


def _compare(got, ref, label, greedy=False):
    """Tokens equal until the first differing position of a row, which must be in the tie
    band; statistics and E rows within tolerance on the agreeing prefix; the tie-band
    cases below the rate bound.  Returns the number of diverged rows."""
    diverged, same = draft_rows(got["tokens"], ref["tokens"], ref["gap"], label)
    for key in ("q_tok", "row_max", "row_sumexp"):
        np.testing.assert_allclose(got[key][same], ref[key][same], rtol=RTOL, err_msg=f"{label} {key}")
    # E at position k depends on tokens before k only: compare where the prefix before k agrees
    before = np.concatenate([np.ones((same.shape[0], 1), bool), same[:, :-1]], axis=1)
    np.testing.assert_allclose(got["E"][before], ref["E"][before], atol=RTOL, err_msg=f"{label} E")
    if greedy:
        np.testing.assert_array_equal(got["q_tok"], 1.0)
    assert_rate(band_cases_draft(ref["gap"]), got["tokens"].size, label)
    return diverged


def test_rnn_pack_is_the_transpose_of_the_recurrent_rows():
    _need_gpu()
    for r, H in [(16, 8), (64, 32), (256, 40), (48, 4)]:
        w = workloads.scaled(workloads.get("tiny"), r=r, H=H)
        W_rnn, _ = workloads.gen_rnn_weights(w)
        Wrec = ds.rnn_pack(ds.as_bf16_tensor(W_rnn), r)
        got = Wrec.view(torch.int16).cpu().numpy().view(np.uint16).reshape(3 * r, 2 * r)
        np.testing.assert_array_equal(got, W_rnn[:2 * r].T)


@pytest.mark.parametrize("name", list(CASES))
def test_rnn_project(name):
    _need_gpu()
    w = CASES[name]
    inp, W_rnn, b_rnn, dev = _setup(w, with_T=False)
    got = ds.rnn_project(dev["h"], dev["W_rnn"], dev["b_rnn"]).cpu().numpy()
    ref = oracle.rnn_project(inp.h, W_rnn, b_rnn)
    mag = np.abs(inp.h).astype(np.float64) @ np.abs(bf16_bits_to_f32(W_rnn)[2 * w.r:]).astype(np.float64)
    np.testing.assert_array_less(np.abs(got - ref), RTOL * (mag + np.abs(b_rnn)) + 1e-12)


# the projection alone on shapes that span its tiles: the full hidden size of the
# 32 x 7, r = 256 workload (40 K chunks, 5 per cluster rank, 6 column tiles, 2 row tiles);
# 144 output columns (a partial second column tile) with a ragged last K chunk (H = 1000);
# 600 rows (5 row tiles) with a K that gives most cluster ranks no chunk at all (H = 12)
PROJECT_SHAPES = {
    "B32_g7_r256_H2560": dict(B=32, gamma=7, r=256, H=2560),
    "B9_g3_r48_H1000": dict(B=9, gamma=3, r=48, H=1000),
    "B300_g2_r16_H12": dict(B=300, gamma=2, r=16, H=12),
}


@pytest.mark.parametrize("name", list(PROJECT_SHAPES))
def test_rnn_project_tiles(name):
    _need_gpu()
    w = workloads.scaled(workloads.get("qwen3_4b_like"), V=1024, **PROJECT_SHAPES[name])
    inp, W_rnn, b_rnn, dev = _setup(w, with_T=False)
    got = ds.rnn_project(dev["h"], dev["W_rnn"], dev["b_rnn"]).cpu().numpy()
    ref = oracle.rnn_project(inp.h, W_rnn, b_rnn)
    assert np.all(np.isfinite(got))
    mag = np.abs(inp.h).astype(np.float64) @ np.abs(bf16_bits_to_f32(W_rnn)[2 * w.r:]).astype(np.float64)
    np.testing.assert_array_less(np.abs(got - ref), RTOL * (mag + np.abs(b_rnn)) + 1e-12)


@pytest.mark.parametrize("greedy", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_draft_rnn(name, greedy):
    _need_gpu()
    w = CASES[name]
    inp, W_rnn, b_rnn, dev = _setup(w, with_T=False)
    ws = ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)
    hp = _cuda(oracle.rnn_project(inp.h, W_rnn, b_rnn), np.float32)
    Wrec = ds.rnn_pack(dev["W_rnn"], w.r)
    out = ds.draft_rnn(dev["U"], dev["W1"], dev["W2"], Wrec, hp, dev["anchor"], w.seed, ws, greedy=greedy)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = oracle.draft_rnn(inp.U, inp.h, inp.W1, inp.W2, W_rnn, b_rnn, inp.anchor, w.seed, greedy=greedy)
    _compare(got, ref, name, greedy)
    # the packed weights give identical outputs
    W2p = ds.pack_w2(dev["W2"])
    out_p = ds.draft_rnn(dev["U"], dev["W1"], W2p, Wrec, hp, dev["anchor"], w.seed, ws, greedy=greedy,
                         packed=True)
    for key in got:
        np.testing.assert_array_equal(got[key], out_p[key].cpu().numpy(), err_msg=key)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_verify_rnn(name):
    _need_gpu()
    w = CASES[name]
    inp, W_rnn, b_rnn, dev = _setup(w)
    ws = ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)
    d = oracle.draft_rnn(inp.U, inp.h, inp.W1, inp.W2, W_rnn, b_rnn, inp.anchor, w.seed)
    rng = np.random.default_rng(w.seed + 600)
    ell = rng.integers(0, w.gamma + 1, size=w.B).astype(np.int32)
    out = ds.verify_rnn(dev["T"], dev["U"], _cuda(d["E"], np.float32), dev["W2"],
                        _cuda(d["tokens"], np.int32), _cuda(d["q_tok"], np.float32),
                        _cuda(d["row_max"], np.float32), _cuda(d["row_sumexp"], np.float32),
                        _cuda(ell, np.int32), w.seed, ws)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = oracle.verify_rnn(inp.T, inp.U, d["E"], inp.W2, d["tokens"], ell, w.seed)
    verify_rows(got, ref, name)
    assert_rate(band_cases_verify(ref), w.B * w.gamma, name)
    assert (got["accept_len"] < ell).sum() > 0 or w.B < 8
    assert ws.status() == 0


def test_full_size_draft_rnn_sampled_requests():
    """qwen3_4b_like at full size in one launch; the oracle recomputes sampled requests."""
    _need_gpu()
    w = workloads.get("qwen3_4b_like")
    inp, W_rnn, b_rnn, dev = _setup(w, with_T=False)
    ws = ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)
    hp = ds.rnn_project(dev["h"], dev["W_rnn"], dev["b_rnn"])
    Wrec = ds.rnn_pack(dev["W_rnn"], w.r)
    got = {k: v.cpu().numpy() for k, v in ds.draft_rnn(dev["U"], dev["W1"], dev["W2"], Wrec, hp,
                                                        dev["anchor"], w.seed, ws).items()}
    assert ws.status() == 0
    assert np.all((got["tokens"] >= 0) & (got["tokens"] < w.V))
    picks = sorted({0, w.B - 1, w.B // 2, 7 % w.B})
    sub = workloads.generate(w, requests=picks, with_T=False)
    ref = oracle.draft_rnn(sub.U, sub.h, sub.W1, sub.W2, W_rnn, b_rnn, sub.anchor, w.seed, req_ids=picks)
    _compare({k: v[picks] for k, v in got.items()}, ref, "qwen3_4b_like")


@pytest.mark.parametrize("sampling", ["gumbel", "greedy"])
@pytest.mark.parametrize("name", ["tiny", "qwen_small", "prod_small"])
def test_rnn_step_end_to_end(name, sampling):
    _need_gpu()
    w = CASES[name]
    inp, W_rnn, b_rnn, dev = _setup(w)
    step = ds.Step(dev, float(inp.b_c), head="rnn", sampling=sampling).run(seed=w.seed)
    got = step.results()
    greedy = sampling == "greedy"
    d = oracle.draft_rnn(inp.U, inp.h, inp.W1, inp.W2, W_rnn, b_rnn, inp.anchor, w.seed, greedy=greedy)
    if _compare({k: got[k] for k in ("tokens", "q_tok", "row_max", "row_sumexp", "E")}, d, name, greedy):
        return
    _, a = oracle.confidence(inp.h, inp.anchor, d["tokens"], inp.W1, inp.w_c, float(inp.b_c))
    np.testing.assert_allclose(got["a"], a, rtol=RTOL)
    # the oracle's chain schedules its own fp32 survivals: the same l unless a stop decision
    # sits within the two chains' rounding, which seeded data does not produce
    ell_r, Bt_r, _ = oracle.schedule(a.astype(np.float32), inp.sps)
    np.testing.assert_array_equal(got["ell"], ell_r)
    assert got["B_total"] == Bt_r
    v = (oracle.verify_greedy(inp.T, d["tokens"], ell_r, w.seed) if greedy else
         oracle.verify_rnn(inp.T, inp.U, d["E"], inp.W2, d["tokens"], ell_r, w.seed))
    verify_rows(got, v, name)
    assert step.ws.status() == 0
