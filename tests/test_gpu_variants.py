"""Parity of the CUDA variants of the step with the CPU oracle: greedy drafting, its
point-mass verification, the asynchronous two-step capacity scheduler and fixed-threshold
truncation.

The bars match the main parity tests.  Token ids, accept lengths and l_r must be
bit-exact, except inside the tie band.  For greedy drafting the band is a top-two logit
gap within 1e-5; for the acceptance test it is |u - p| within 1e-5.  Row statistics must
agree within 1e-5 relative.  q_tok of a greedy draft must be exactly 1.  The schedulers
are integer and fixed-point work, so they must be bit-exact.
"""
import numpy as np
import pytest

import oracle
import workloads
from _parity import (assert_rate, band_cases_draft, band_cases_verify, draft_rows, draft_stats,
                     verify_rows)

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


def _ws(w):
    return ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)


def _compare_greedy(got, ref, label):
    """Tokens equal until the first differing position of a row, which must be in the tie
    band; row statistics within RTOL on the agreeing prefix; the tie-band cases of the
    batch below the rate bound.  Returns the number of diverged rows."""
    diverged, same = draft_rows(got["tokens"], ref["tokens"], ref["gap"], label)
    draft_stats(got, ref, same, keys=("row_max", "row_sumexp"), label=label)
    np.testing.assert_array_equal(got["q_tok"], 1.0)
    assert_rate(band_cases_draft(ref["gap"]), got["tokens"].size, label)
    return diverged


# ------------------------------------------------------------------------ greedy draft

@pytest.mark.parametrize("name", list(CASES))
def test_draft_greedy(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w, with_T=False)
    dev = ds.to_device(inp)
    ws = _ws(w)
    got = {k: v.cpu().numpy() for k, v in ds.draft_greedy(dev["U"], dev["W1"], dev["W2"],
                                                           dev["anchor"], ws).items()}
    ref = oracle.draft_greedy(inp.U, inp.W1, inp.W2, inp.anchor)
    _compare_greedy(got, ref, name)
    # the packed weights give identical outputs
    W2p = ds.pack_w2(dev["W2"])
    got_p = {k: v.cpu().numpy() for k, v in ds.draft_greedy(dev["U"], dev["W1"], W2p,
                                                             dev["anchor"], ws, packed=True).items()}
    for key in got:
        np.testing.assert_array_equal(got[key], got_p[key], err_msg=key)
    assert ws.status() == 0


def test_draft_greedy_ties_go_to_the_smallest_index():
    # equal largest logits in different tiles, lanes and CTAs of the vocabulary
    _need_gpu()
    B, gamma, V, r = 3, 2, 4096, 16
    U = np.zeros((B, gamma, V), np.float32)
    U[0, :, [5, 6, 1000, 4095]] = 3.0
    U[1, :, [4095, 2048]] = 3.0
    U[2, 0, [129, 128 + 4]] = 3.0
    U[2, 1, [700, 3000]] = 3.0
    W1 = np.zeros((V, r), np.uint16)
    W2 = np.zeros((r, V), np.uint16)
    ws = ds.Workspace(B, gamma, V, r)
    d = ds.draft_greedy(_cuda(U, np.float32), ds.as_bf16_tensor(W1), ds.as_bf16_tensor(W2),
                        _cuda(np.zeros(B), np.int32), ws)
    assert d["tokens"].cpu().numpy().tolist() == [[5, 5], [2048, 2048], [129, 700]]
    assert ws.status() == 0


@pytest.mark.parametrize("name", ["qwen3_4b_like", "scheduler_stress"])
def test_full_size_draft_greedy_sampled_requests(name):
    """Full size in the benchmark's launch configuration; the oracle recomputes the whole
    block of a few sampled requests."""
    _need_gpu()
    w = workloads.get(name)
    inp = workloads.generate(w, with_T=False)
    dev = ds.to_device(inp)
    ws = _ws(w)
    got = {k: v.cpu().numpy() for k, v in ds.draft_greedy(dev["U"], dev["W1"], dev["W2"],
                                                           dev["anchor"], ws).items()}
    assert ws.status() == 0
    assert np.all((got["tokens"] >= 0) & (got["tokens"] < w.V))
    assert np.all(got["row_sumexp"] >= 1)
    picks = sorted({0, w.B - 1, w.B // 2, 7 % w.B})
    sub = workloads.generate(w, requests=picks, with_T=False)
    ref = oracle.draft_greedy(sub.U, sub.W1, sub.W2, sub.anchor)
    _compare_greedy({k: v[picks] for k, v in got.items()}, ref, name)


# ---------------------------------------------------------------------- greedy verify

@pytest.mark.parametrize("name", list(CASES))
def test_verify_greedy(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w)
    dev = ds.to_device(inp)
    ws = _ws(w)
    d = oracle.draft_greedy(inp.U, inp.W1, inp.W2, inp.anchor)
    rng = np.random.default_rng(w.seed + 300)
    ell = rng.integers(0, w.gamma + 1, size=w.B).astype(np.int32)
    out = ds.verify_greedy(dev["T"], _cuda(d["tokens"], np.int32), _cuda(ell, np.int32), w.seed, ws)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = oracle.verify_greedy(inp.T, d["tokens"], ell, w.seed)
    verify_rows(got, ref, name)
    assert_rate(band_cases_verify(ref), w.B * w.gamma, name)
    np.testing.assert_array_equal(got["n_out"], got["accept_len"] + 1)
    # a correction is never the rejected draft token
    for i in range(w.B):
        j = got["accept_len"][i]
        if j < ell[i]:
            assert got["out_tokens"][i, j] != d["tokens"][i, j]
    assert ws.status() == 0


def test_verify_greedy_rejects_and_corrects_on_a_peaked_target():
    # target rows that put almost all mass on another token: nearly every first position
    # rejects, and the correction is that token or another one, never the draft's
    _need_gpu()
    B, gamma, V = 64, 3, 1024
    rng = np.random.default_rng(31)
    T = rng.normal(0, 1, size=(B, gamma + 1, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    peak = (tokens + 17) % V
    for b in range(B):
        T[b, 0, peak[b, 0]] = 30.0
    ell = np.full(B, gamma, np.int32)
    ws = ds.Workspace(B, gamma, V, 16)
    got = {k: v.cpu().numpy() for k, v in ds.verify_greedy(
        _cuda(T, np.float32), _cuda(tokens, np.int32), _cuda(ell, np.int32), 9, ws).items()}
    ref = oracle.verify_greedy(T, tokens, ell, 9)
    for key in ("accept_len", "out_tokens", "n_out"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    assert np.all(got["accept_len"] == 0)
    assert np.all(got["out_tokens"][:, 0] == peak[:, 0])
    assert ws.status() == 0


# ------------------------------------------------------------------ async scheduler

def _survival(rng, R, gamma, lo=0.2):
    return np.cumprod(rng.uniform(lo, 1.0, size=(R, gamma)), axis=1).astype(np.float32)


@pytest.mark.parametrize("name", list(CASES))
def test_schedule_async(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w, with_T=False)
    ws = _ws(w)
    rng = np.random.default_rng(w.seed + 400)
    a = _survival(rng, w.B, w.gamma)
    a[0, :] = a[0, 0]
    if w.B > 2:
        a[1, :] = a[0, :]
    a_d, sps_d = _cuda(a, np.float32), _cuda(inp.sps, np.float32)
    N = w.B * w.gamma
    n_star = oracle.schedule(a, inp.sps)[1] - w.B
    for K in [None, -1, 0, 1, N // 3, n_star, N, N + 5]:
        K_in = None if K is None else _cuda([K], np.int32)
        K_out = _cuda([-7], np.int32)
        ell, Bt, th = ds.schedule_async(a_d, sps_d, K_in, K_out, ws)
        ell_r, Bt_r, th_r, ko_r = oracle.schedule_async(a, inp.sps, -1 if K is None else K)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_r, err_msg=str(K))
        assert int(Bt.item()) == Bt_r and float(th.item()) == th_r and int(K_out.item()) == ko_r
    # K_in and K_out the same word: read first, then overwritten with this step's count
    k = _cuda([N // 2], np.int32)
    ell, Bt, _ = ds.schedule_async(a_d, sps_d, k, k, ws)
    assert int(Bt.item()) == w.B + N // 2 and int(k.item()) == n_star
    assert ws.status() == 0


def test_schedule_async_ring_pipeline():
    _need_gpu()
    rng = np.random.default_rng(41)
    R, gamma, steps = 96, 7, 8
    sps = (1.0 / (1.0 + 0.004 * np.maximum(0, np.arange(R * (gamma + 1) + 1) - 200))).astype(np.float32)
    ring = ds.CapacityRing()
    ws = ds.Workspace(R, gamma, 1024, 16)
    want_ring = [-1, -1]
    for t in range(steps):
        a = _survival(rng, R, gamma, lo=0.1 + 0.15 * (t % 4))
        ell, Bt, th = ds.schedule_async(_cuda(a, np.float32), _cuda(sps, np.float32),
                                        ring.slot(t), ring.slot(t), ws)
        ell_r, Bt_r, th_r, ko_r = oracle.schedule_async(a, sps, want_ring[t % 2])
        want_ring[t % 2] = ko_r
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_r, err_msg=str(t))
        assert int(Bt.item()) == Bt_r and float(th.item()) == th_r
        assert ring.slots.cpu().numpy().tolist() == want_ring
    assert ws.status() == 0


def test_schedule_async_large_batch_uses_the_radix_sort():
    _need_gpu()
    rng = np.random.default_rng(42)
    R, gamma = 1024, 16                      # 16384 items: radix path
    a = _survival(rng, R, gamma, lo=0.5)
    n = np.arange(R * (gamma + 1) + 1)
    sps = (1.0 / (1.0 + np.maximum(0, n - 512) / 512.0)).astype(np.float32)
    ws = ds.Workspace(R, gamma, 1024, 16)
    for K in [-1, 0, 777, 16384]:
        K_in, K_out = _cuda([K], np.int32), _cuda([0], np.int32)
        ell, Bt, th = ds.schedule_async(_cuda(a, np.float32), _cuda(sps, np.float32), K_in, K_out, ws)
        ell_r, Bt_r, th_r, ko_r = oracle.schedule_async(a, sps, K)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_r)
        assert int(Bt.item()) == Bt_r and float(th.item()) == th_r and int(K_out.item()) == ko_r
    assert ws.status() == 0


# ---------------------------------------------------------------- threshold truncation

@pytest.mark.parametrize("R,gamma", [(1, 1), (5, 3), (300, 2), (1024, 16), (40, 32), (3000, 7)])
def test_schedule_threshold(R, gamma):
    _need_gpu()
    rng = np.random.default_rng(R + gamma)
    a = _survival(rng, R, gamma)
    a[::5] = rng.uniform(0, 1, size=a[::5].shape).astype(np.float32)   # not monotone
    a[1::7, 0] = np.float32(0.5)                                       # exactly at the threshold
    a[2::11, -1] = np.nan
    a_d = _cuda(a, np.float32)
    for th in [-1.0, 0.0, 0.25, 0.5, 0.9, 1.0]:
        ell, Bt = ds.schedule_threshold(a_d, th)
        ell_r, Bt_r = oracle.schedule_threshold(a, th)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_r, err_msg=str(th))
        assert int(Bt.item()) == Bt_r


# ------------------------------------------------------------------- whole step chains

@pytest.mark.parametrize("name", ["tiny", "qwen_small", "prod_small"])
@pytest.mark.parametrize("scheduler", ["threshold", "async"])
def test_greedy_step_end_to_end(name, scheduler):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w)
    step = ds.Step(ds.to_device(inp), float(inp.b_c), sampling="greedy", scheduler=scheduler,
                   threshold=0.4)
    step.run(seed=w.seed, t=0)
    got = step.results()
    d = oracle.draft_greedy(inp.U, inp.W1, inp.W2, inp.anchor)
    if _compare_greedy({k: got[k] for k in ("tokens", "q_tok", "row_max", "row_sumexp")}, d, name):
        return
    _, a = oracle.confidence(inp.h, inp.anchor, d["tokens"], inp.W1, inp.w_c, float(inp.b_c))
    np.testing.assert_allclose(got["a"], a, rtol=RTOL)
    # the oracle's chain schedules its own survivals (fp32): the same l unless a decision
    # sits within the two chains' rounding, which seeded data does not produce
    a32 = a.astype(np.float32)
    if scheduler == "threshold":
        ell_r, Bt_r = oracle.schedule_threshold(a32, 0.4)
    else:
        ell_r, Bt_r, _, _ = oracle.schedule_async(a32, inp.sps, -1)
    np.testing.assert_array_equal(got["ell"], ell_r)
    assert got["B_total"] == Bt_r
    v = oracle.verify_greedy(inp.T, d["tokens"], ell_r, w.seed)
    verify_rows(got, v, name)
    assert step.ws.status() == 0
