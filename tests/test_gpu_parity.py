"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars (the tolerances the method's statement fixes):
  * token ids, accept lengths, l_r: bit-exact, except inside the tie band -- the top-two
    Gumbel scores within 1e-5 of each other, or |u - p/q| within 1e-5 -- and such cases
    must stay below 1e-4 of the positions;
  * probabilities and confidences (q_tok, row_max, row_sumexp, c, a): within 1e-5
    relative in fp32.
Each call is fed the oracle's upstream outputs (never the other way round), so that every
call is compared on identical inputs; the end-to-end chain is compared separately.  The
rules (where the tie band is checked, the rate bound) are in ``_parity``.
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


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# small cases that span several 128-row vocabulary tiles, a ragged last tile, batch
# chunks of the tensor-core contraction (B > 256), the one-pass 256-row contraction
# (128 < B <= 256), and every Markov rank shape
CASES = {
    "tiny": workloads.get("tiny"),
    "qwen_small": workloads.scaled(workloads.get("qwen3_4b_like"), B=5, gamma=3, V=904, r=64, H=32),
    "prod_small": workloads.scaled(workloads.get("production"), B=40, gamma=5, V=2056, r=256, H=64),
    "long_small": workloads.scaled(workloads.get("long_block"), B=7, gamma=15, V=1032, r=256, H=16,
                                   noise_std=lambda k: 0.5 + 1.5 * (k - 1) / 14.0),
    "wide_batch": workloads.scaled(workloads.get("scheduler_stress"), B=300, gamma=2, V=520, r=128, H=8),
    "mid_batch": workloads.scaled(workloads.get("production"), B=200, gamma=3, V=1160, r=256, H=16),
}


def _dev(inp):
    return ds.to_device(inp, "cuda")


def _ws(w):
    return ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)


@pytest.mark.parametrize("name", list(CASES))
def test_markov_bias(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    rng = np.random.default_rng(5)
    prev = rng.integers(0, w.V, size=w.B).astype(np.int32)
    prev[::7] = -1
    got = ds.markov_bias(dev["W1"], dev["W2"], torch.from_numpy(prev).cuda(), ws).cpu().numpy()
    ref = oracle.markov_bias(inp.W1, inp.W2, prev)
    W1f = workloads.bf16_bits_to_f32(inp.W1).astype(np.float64)
    W2f = workloads.bf16_bits_to_f32(inp.W2).astype(np.float64)
    mag = np.abs(W1f[np.maximum(prev, 0)]) @ np.abs(W2f)
    mag[prev < 0] = 0
    np.testing.assert_array_less(np.abs(got - ref), RTOL * mag + 1e-12)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_draft(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    got = {k: v.cpu().numpy() for k, v in ds.draft(dev["U"], dev["W1"], dev["W2"], dev["anchor"],
                                                    w.seed, ws).items()}
    ref = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    _, same = draft_rows(got["tokens"], ref["tokens"], ref["gap"], name)
    draft_stats(got, ref, same, label=name)
    assert_rate(band_cases_draft(ref["gap"]), got["tokens"].size, name)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_confidence(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    d = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    tok = torch.from_numpy(d["tokens"]).cuda()
    c, a = ds.confidence(dev["h"], dev["anchor"], tok, dev["W1"], dev["w_c"], float(inp.b_c), ws)
    c_ref, a_ref = oracle.confidence(inp.h, inp.anchor, d["tokens"], inp.W1, inp.w_c, float(inp.b_c))
    np.testing.assert_allclose(c.cpu().numpy(), c_ref, rtol=RTOL)
    np.testing.assert_allclose(a.cpu().numpy(), a_ref, rtol=RTOL)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_schedule(name):
    _need_gpu()
    w = CASES[name]
    if w.B * w.gamma > 16384:
        pytest.skip("beyond the one-CTA scheduler")
    inp = workloads.generate(w, with_T=False)
    ws = _ws(w)
    rng = np.random.default_rng(w.seed)
    a = np.cumprod(rng.uniform(0.2, 1.0, size=(w.B, w.gamma)), axis=1).astype(np.float32)
    a[0, :] = a[0, 0]                            # exact ties inside a request
    if w.B > 2:
        a[1, :] = a[0, :]                        # exact ties across requests
    ell, Bt, th = ds.schedule(torch.from_numpy(a).cuda(), torch.from_numpy(inp.sps).cuda(), ws)
    ell_ref, Bt_ref, th_ref = oracle.schedule(a, inp.sps)
    np.testing.assert_array_equal(ell.cpu().numpy(), ell_ref)
    assert int(Bt.item()) == Bt_ref
    assert float(th.item()) == th_ref
    assert ws.status() == 0


def test_schedule_random_tables_and_sizes():
    _need_gpu()
    rng = np.random.default_rng(11)
    for R, gamma in [(1, 1), (1, 7), (3, 5), (33, 4), (100, 16), (1024, 16), (700, 23)]:
        if R * gamma > 16384:
            continue
        a = np.cumprod(rng.uniform(0.0, 1.0, size=(R, gamma)) ** 0.3, axis=1).astype(np.float32)
        n = np.arange(R * (gamma + 1) + 1)
        for sps in [1.0 / (1.0 + rng.uniform(0.001, 0.05) * n),
                    1.0 / (1.0 + np.maximum(0, n - R * 2) / (R + 1.0)),
                    rng.uniform(0.5, 1.0, size=n.size)]:
            sps = sps.astype(np.float32)
            ws = ds.Workspace(R, gamma, 8, 16, 0)
            ell, Bt, th = ds.schedule(torch.from_numpy(a).cuda(), torch.from_numpy(sps).cuda(), ws)
            ell_ref, Bt_ref, th_ref = oracle.schedule(a, sps)
            np.testing.assert_array_equal(ell.cpu().numpy(), ell_ref)
            assert int(Bt.item()) == Bt_ref and float(th.item()) == th_ref


def test_schedule_radix_path_edge_values():
    """More items than the scheduler's threads (the radix path): exact ties inside and
    across requests, survivals of 0, NaN, 1 and above, subnormal, and the two smallest
    fixed-point values (A = 0 and A = 1, which differ in the key's 33rd bit)."""
    _need_gpu()
    rng = np.random.default_rng(5)
    R, gamma = 600, 4                                    # 2400 items
    a = np.cumprod(rng.uniform(0.0, 1.0, size=(R, gamma)) ** 0.2, axis=1).astype(np.float32)
    a[10:60, :] = a[5, :]                                # exact ties across requests
    a[70, :] = 0.0
    a[71, :] = np.float32(np.nan)
    a[72, :] = np.float32(1.0)
    a[73, :] = np.float32(1.5)
    a[74, :] = np.float32(1e-45)                         # subnormal: A = 0
    a[75, :] = np.float32(2.0 ** -32)                    # A = 1
    a[76, :] = np.float32(2.0 ** -33)                    # rounds half up to A = 1
    a[77, :] = np.float32(np.nextafter(np.float32(2.0 ** -33), np.float32(0)))   # A = 0
    n = np.arange(R * (gamma + 1) + 1)
    for sps in [1.0 / (1.0 + 0.0005 * n), 1.0 / (1.0 + np.maximum(0, n - R) / (4.0 * R))]:
        sps = sps.astype(np.float32)
        ws = ds.Workspace(R, gamma, 8, 16, 0)
        ell, Bt, th = ds.schedule(torch.from_numpy(a).cuda(), torch.from_numpy(sps).cuda(), ws)
        ell_ref, Bt_ref, th_ref = oracle.schedule(a, sps)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_ref)
        assert int(Bt.item()) == Bt_ref and float(th.item()) == th_ref
        # a capacity that stops inside the zero-survival tail: the order of the last items
        # (A = 0 after A = 1, then request order) decides which requests keep a position
        for K in (R * gamma - 7, R * gamma - 13):
            K_in = torch.tensor([K], dtype=torch.int32, device="cuda")
            K_out = torch.zeros(1, dtype=torch.int32, device="cuda")
            ell, Bt, th = ds.schedule_async(torch.from_numpy(a).cuda(), torch.from_numpy(sps).cuda(),
                                            K_in, K_out, ws)
            ell_r, Bt_r, th_r, ko_r = oracle.schedule_async(a, sps, K)
            np.testing.assert_array_equal(ell.cpu().numpy(), ell_r)
            assert int(Bt.item()) == Bt_r and float(th.item()) == th_r and int(K_out.item()) == ko_r
        assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_verify(name):
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w)
    dev = _dev(inp)
    ws = _ws(w)
    d = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    rng = np.random.default_rng(w.seed + 100)
    ell = rng.integers(0, w.gamma + 1, size=w.B).astype(np.int32)
    cuda = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x, dtype=dt)).cuda()
    out = ds.verify(dev["T"], dev["U"], dev["W1"], dev["W2"], dev["anchor"],
                    cuda(d["tokens"], np.int32), cuda(d["q_tok"], np.float32),
                    cuda(d["row_max"], np.float32), cuda(d["row_sumexp"], np.float32),
                    cuda(ell, np.int32), w.seed, ws)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = oracle.verify(inp.T, inp.U, inp.W1, inp.W2, inp.anchor, d["tokens"], ell, w.seed)
    verify_rows(got, ref, name)
    assert_rate(band_cases_verify(ref), w.B * w.gamma, name)
    np.testing.assert_array_equal(got["n_out"], got["accept_len"] + 1)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_step_end_to_end(name):
    """The GPU chain (each call consuming the GPU's own upstream outputs) against the
    oracle's chain on the same inputs: equal while no decision falls in the tie band."""
    _need_gpu()
    w = CASES[name]
    if w.B * w.gamma > 16384:
        pytest.skip("beyond the one-CTA scheduler")
    inp = workloads.generate(w)
    step = ds.Step(_dev(inp), float(inp.b_c)).run(seed=w.seed)
    got = step.results()
    ref = oracle.step(inp, seed=w.seed)
    diverged, _ = draft_rows(got["tokens"], ref["draft"]["tokens"], ref["draft"]["gap"], name)
    if diverged == 0:
        np.testing.assert_allclose(got["c"], ref["c"], rtol=RTOL)
        np.testing.assert_allclose(got["a"], ref["a"], rtol=RTOL)
        # the two chains schedule survivals computed in fp32 and fp64: the same l unless a
        # stop decision sits within their rounding, which seeded data does not produce
        np.testing.assert_array_equal(got["ell"], ref["ell"])
        assert got["B_total"] == ref["B_total"]
        verify_rows(got, ref["verify"], name)
    assert step.ws.status() == 0


def test_device_check_reports_bad_token_ids():
    _need_gpu()
    w = CASES["tiny"]
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    bad = dev["anchor"].clone()
    bad[1] = w.V + 5
    ds.draft(dev["U"], dev["W1"], dev["W2"], bad, w.seed, ws)
    assert ws.status() == 5          # DSPARK_ERR_DEVICE_CHECK, read and cleared
    assert ws.status() == 0


# ------------------------------------------------------------- full-size workloads

FULL = ["qwen3_4b_like", "production", "long_block", "scheduler_stress"]


def _to(x, dt):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=dt)).cuda()


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_request(name):
    """Every call of the benchmarked step at full size, in the benchmark's launch
    configuration (packed W2, the scheduler in the confidence kernel's last CTA, the packed
    verification), against the oracle on every request.  Each call gets the oracle's
    upstream outputs; the tie-band cases of the whole batch are counted and held below
    1e-4 of its positions.  The captured step (what the benchmark replays: the draft,
    confidence and schedule in one launch, then the verification) must then give the
    per-call results wherever its inputs coincide with them."""
    _need_gpu()
    w = workloads.get(name)
    inp = workloads.generate(w)
    n_pos = w.B * w.gamma
    d = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    c_ref, a_ref = oracle.confidence(inp.h, inp.anchor, d["tokens"], inp.W1, inp.w_c, float(inp.b_c))
    a32 = a_ref.astype(np.float32)
    ell_ref, Bt_ref, th_ref = oracle.schedule(a32, inp.sps)
    v = oracle.verify(inp.T, inp.U, inp.W1, inp.W2, inp.anchor, d["tokens"], ell_ref, w.seed)

    dev = _dev(inp)
    ws = _ws(w)
    W2p = ds.pack_w2(dev["W2"])
    # draft
    gd = {k: t.cpu().numpy() for k, t in ds.draft_packed(dev["U"], dev["W1"], W2p, dev["anchor"],
                                                          w.seed, ws).items()}
    diverged, same = draft_rows(gd["tokens"], d["tokens"], d["gap"], name)
    draft_stats(gd, d, same, label=name)
    # confidence + scheduler (one launch), fed the oracle's tokens
    tok = _to(d["tokens"], np.int32)
    (c, a), (ell, Bt, th) = ds.confidence_schedule(dev["h"], dev["anchor"], tok, dev["W1"], dev["w_c"],
                                                   float(inp.b_c), dev["sps"], ws)
    np.testing.assert_allclose(c.cpu().numpy(), c_ref, rtol=RTOL)
    np.testing.assert_allclose(a.cpu().numpy(), a_ref, rtol=RTOL)
    ell_s, Bt_s, th_s = ds.schedule(a, dev["sps"], ws)      # the same a, the standalone kernel
    np.testing.assert_array_equal(ell.cpu().numpy(), ell_s.cpu().numpy())
    assert int(Bt.item()) == int(Bt_s.item()) and float(th.item()) == float(th_s.item())
    # the scheduler on the oracle's fp32 survivals: exact
    ell_o, Bt_o, th_o = ds.schedule(_to(a32, np.float32), dev["sps"], ws)
    np.testing.assert_array_equal(ell_o.cpu().numpy(), ell_ref)
    assert int(Bt_o.item()) == Bt_ref and float(th_o.item()) == th_ref
    # verification of the oracle's tokens with the oracle's lengths
    out = ds.verify_packed(dev["T"], dev["U"], dev["W1"], W2p, dev["anchor"], tok,
                           _to(d["q_tok"], np.float32), _to(d["row_max"], np.float32),
                           _to(d["row_sumexp"], np.float32), _to(ell_ref, np.int32), w.seed, ws)
    gv = {k: t.cpu().numpy() for k, t in out.items()}
    v_div = verify_rows(gv, v, name)
    np.testing.assert_array_equal(gv["n_out"], gv["accept_len"] + 1)
    assert ws.status() == 0
    cases = band_cases_draft(d["gap"]) + band_cases_verify(v)
    print(f"\n{name}: {n_pos} positions, tie-band cases {cases} (draft {band_cases_draft(d['gap'])}, "
          f"verify {band_cases_verify(v)}), diverged draft rows {diverged}, verify rows {v_div}, "
          f"mean l {ell_ref.mean():.2f}, mean accept {v['accept_len'].mean():.2f}")
    assert_rate(cases, n_pos, name)

    # the step as the benchmark captures and replays it
    step = ds.Step(dev, float(inp.b_c), ws=ws, W2p=W2p)
    g = step.capture([w.seed])[0]
    g.replay()
    torch.cuda.synchronize()
    st = step.results()
    assert step.ws.status() == 0
    np.testing.assert_array_equal(st["tokens"], gd["tokens"])
    for key in ("q_tok", "row_max", "row_sumexp"):
        np.testing.assert_array_equal(st[key], gd[key], err_msg=key)
    if diverged == 0:
        # the step computes confidence inside the draft launch (another summation order)
        np.testing.assert_allclose(st["c"], c_ref, rtol=RTOL)
        np.testing.assert_allclose(st["a"], a_ref, rtol=RTOL)
        ell_st, Bt_st, th_st = ds.schedule(torch.from_numpy(st["a"]).cuda(), dev["sps"], ws)
        np.testing.assert_array_equal(st["ell"], ell_st.cpu().numpy())
        assert st["B_total"] == int(Bt_st.item())
        if np.array_equal(st["ell"], ell_ref):
            # the step verifies with its own fp32 draft statistics: the oracle's outcomes
            # outside the tie band
            verify_rows(st, v, name + " (captured step)")


@pytest.mark.parametrize("name", list(CASES))
def test_draft_packed_matches_draft(name):
    """The packed-weights draft runs the same kernel arithmetic: identical outputs."""
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    W2p = ds.pack_w2(dev["W2"])
    assert W2p.numel() * 2 == ds.lib().dspark_packed_w2_bytes(w.V, w.r)
    a = {k: v.cpu().numpy() for k, v in ds.draft(dev["U"], dev["W1"], dev["W2"], dev["anchor"],
                                                  w.seed, ws).items()}
    b = {k: v.cpu().numpy() for k, v in ds.draft_packed(dev["U"], dev["W1"], W2p, dev["anchor"],
                                                         w.seed, ws).items()}
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_verify_packed_matches_verify(name):
    """The packed-weights verification feeds the same operands to the same contraction:
    identical outputs."""
    _need_gpu()
    w = CASES[name]
    inp = workloads.generate(w)
    dev = _dev(inp)
    ws = _ws(w)
    W2p = ds.pack_w2(dev["W2"])
    d = ds.draft(dev["U"], dev["W1"], dev["W2"], dev["anchor"], w.seed, ws)
    rng = np.random.default_rng(w.seed + 200)
    ell = torch.from_numpy(rng.integers(0, w.gamma + 1, size=w.B).astype(np.int32)).cuda()
    args = (d["tokens"], d["q_tok"], d["row_max"], d["row_sumexp"], ell, w.seed, ws)
    a = {k: v.cpu().numpy() for k, v in ds.verify(dev["T"], dev["U"], dev["W1"], dev["W2"],
                                                   dev["anchor"], *args).items()}
    b = {k: v.cpu().numpy() for k, v in ds.verify_packed(dev["T"], dev["U"], dev["W1"], W2p,
                                                          dev["anchor"], *args).items()}
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    assert ws.status() == 0


def test_pack_layout_matches_its_definition():
    """dspark_pack_w2 against the layout the header states, rebuilt with numpy."""
    _need_gpu()
    for V, r in [(904, 64), (520, 128), (1032, 256), (1000, 16), (264, 48)]:
        rng = np.random.default_rng(V + r)
        W2 = rng.integers(0, 2**16, size=(r, V), dtype=np.uint16)
        W2d = torch.from_numpy(W2.view(np.int16)).cuda().view(torch.bfloat16)
        got = ds.pack_w2(W2d).cpu().view(torch.int16).numpy().view(np.uint16)
        kc = 64 if r % 64 == 0 else 32 if r % 32 == 0 else 16
        n_tiles = -(-V // 128)
        Wpad = np.zeros((r, n_tiles * 128), np.uint16)
        Wpad[:, :V] = W2
        want = np.empty((n_tiles, r // kc, 2, kc, 8, 8), np.uint16)
        for kl in range(kc):
            for s in range(8):
                c = s ^ (kl % 8)
                for t in range(n_tiles):
                    for h in range(2):
                        v = t * 128 + 64 * h + 8 * c
                        want[t, :, h, kl, s, :] = Wpad[kl::kc, v:v + 8].reshape(r // kc, 8)
        np.testing.assert_array_equal(got, want.reshape(-1), err_msg=f"V={V} r={r}")


@pytest.mark.parametrize("name", list(CASES))
def test_confidence_schedule_fused_matches_the_two_calls(name):
    """The confidence kernel's last CTA runs the scheduler: identical c, a, l, B, Theta."""
    _need_gpu()
    w = CASES[name]
    if w.B * w.gamma > 16384:
        pytest.skip("beyond the one-CTA scheduler")
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    d = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    tok = torch.from_numpy(d["tokens"]).cuda()
    args = (dev["h"], dev["anchor"], tok, dev["W1"], dev["w_c"], float(inp.b_c))
    c1, a1 = ds.confidence(*args, ws)
    ell1, Bt1, th1 = ds.schedule(a1, dev["sps"], ws)
    for _ in range(2):          # twice: the CTA counter is back at zero after a call
        (c2, a2), (ell2, Bt2, th2) = ds.confidence_schedule(*args, dev["sps"], ws)
        np.testing.assert_array_equal(c1.cpu().numpy(), c2.cpu().numpy())
        np.testing.assert_array_equal(a1.cpu().numpy(), a2.cpu().numpy())
        np.testing.assert_array_equal(ell1.cpu().numpy(), ell2.cpu().numpy())
        assert int(Bt1.item()) == int(Bt2.item()) and float(th1.item()) == float(th2.item())
    ell_r, Bt_r, th_r = oracle.schedule(a2.cpu().numpy(), inp.sps)
    np.testing.assert_array_equal(ell2.cpu().numpy(), ell_r)
    assert ws.status() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_draft_confidence_schedule_in_one_launch(name):
    """The fused first three calls: the draft identical to dspark_draft_packed's, the
    confidence and survival of the drafted tokens within the tolerance of the confidence
    call (and of the oracle), the schedule that of the scheduler on the fused survivals."""
    _need_gpu()
    w = CASES[name]
    if w.B * w.gamma > 16384:
        pytest.skip("beyond the one-CTA scheduler")
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    W2p = ds.pack_w2(dev["W2"])
    d1 = {k: t.cpu().numpy() for k, t in ds.draft_packed(dev["U"], dev["W1"], W2p, dev["anchor"],
                                                          w.seed, ws).items()}
    for _ in range(2):       # twice: nothing in the workspace carries over
        d2, (c2, a2), (ell2, Bt2, th2) = ds.draft_confidence_schedule(
            dev["U"], dev["W1"], W2p, dev["anchor"], dev["h"], dev["w_c"], float(inp.b_c), dev["sps"],
            w.seed, ws)
        for key in d1:
            np.testing.assert_array_equal(d2[key].cpu().numpy(), d1[key], err_msg=key)
        c1, a1 = ds.confidence(dev["h"], dev["anchor"], d2["tokens"], dev["W1"], dev["w_c"],
                               float(inp.b_c), ws)
        np.testing.assert_allclose(c2.cpu().numpy(), c1.cpu().numpy(), rtol=RTOL)
        np.testing.assert_allclose(a2.cpu().numpy(), a1.cpu().numpy(), rtol=RTOL)
        ell1, Bt1, th1 = ds.schedule(a2, dev["sps"], ws)
        np.testing.assert_array_equal(ell2.cpu().numpy(), ell1.cpu().numpy())
        assert int(Bt2.item()) == int(Bt1.item()) and float(th2.item()) == float(th1.item())
    # against the oracle on its own chain (equal while no draft decision is in the band)
    ref = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    if draft_rows(d1["tokens"], ref["tokens"], ref["gap"], name)[0] == 0:
        c_ref, a_ref = oracle.confidence(inp.h, inp.anchor, ref["tokens"], inp.W1, inp.w_c, float(inp.b_c))
        np.testing.assert_allclose(c2.cpu().numpy(), c_ref, rtol=RTOL)
        np.testing.assert_allclose(a2.cpu().numpy(), a_ref, rtol=RTOL)
    assert ws.status() == 0


def test_first_launch_ranks_more_items_than_threads_per_cta():
    """The first launch's grid ranking with shares larger than a CTA's threads (1000
    requests x 2 positions on a 5-tile vocabulary: a grid of 5 CTAs, 400 items each): the
    schedule equals the scheduler's on the same survivals."""
    _need_gpu()
    w = workloads.scaled(workloads.get("scheduler_stress"), B=1000, gamma=2, V=520, r=128, H=8)
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    W2p = ds.pack_w2(dev["W2"])
    d, (c, a), (ell, Bt, th) = ds.draft_confidence_schedule(
        dev["U"], dev["W1"], W2p, dev["anchor"], dev["h"], dev["w_c"], float(inp.b_c), dev["sps"],
        w.seed, ws)
    ell1, Bt1, th1 = ds.schedule(a, dev["sps"], ws)
    np.testing.assert_array_equal(ell.cpu().numpy(), ell1.cpu().numpy())
    assert int(Bt.item()) == int(Bt1.item()) and float(th.item()) == float(th1.item())
    ell_r, Bt_r, th_r = oracle.schedule(a.cpu().numpy(), inp.sps)
    np.testing.assert_array_equal(ell.cpu().numpy(), ell_r)
    assert int(Bt.item()) == Bt_r and float(th.item()) == th_r
    assert ws.status() == 0


@pytest.mark.parametrize("B,gamma,V", [(12, 32, 1664), (8, 4, 1024), (3, 2, 65536), (2, 1, 8192),
                                        (256, 16, 1024), (241, 17, 1024)])
def test_first_launch_scheduler_placements(B, gamma, V):
    """The first launch schedules up to 384 items in the confidence warps of the CTAs that
    hold no request (one such CTA ranking all 384 items; 149 of them sharing 6 items, most
    shares empty), or, with no such CTA (as many CTAs as requests), in CTA 0 after the last
    position; up to 4096 items with the whole grid ranking (exactly 4096 here), beyond that
    with the scheduler kernel after the launch (4097): the schedule equals the scheduler's
    on the same survivals, and the oracle's."""
    _need_gpu()
    w = workloads.scaled(workloads.get("qwen3_4b_like"), B=B, gamma=gamma, V=V, r=64, H=16)
    inp = workloads.generate(w, with_T=False)
    dev = _dev(inp)
    ws = _ws(w)
    W2p = ds.pack_w2(dev["W2"])
    for seed in (w.seed, w.seed + 1):
        d, (c, a), (ell, Bt, th) = ds.draft_confidence_schedule(
            dev["U"], dev["W1"], W2p, dev["anchor"], dev["h"], dev["w_c"], float(inp.b_c),
            dev["sps"], seed, ws)
        ell1, Bt1, th1 = ds.schedule(a, dev["sps"], ws)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell1.cpu().numpy())
        assert int(Bt.item()) == int(Bt1.item()) and float(th.item()) == float(th1.item())
        ell_r, Bt_r, th_r = oracle.schedule(a.cpu().numpy(), inp.sps)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_r)
        assert int(Bt.item()) == Bt_r and float(th.item()) == th_r
    assert ws.status() == 0


def test_schedule_with_exactly_one_block_of_items():
    """R * gamma equal to the scheduler's thread count (the last SPS entry is staged too)."""
    _need_gpu()
    rng = np.random.default_rng(12)
    for R, gamma in [(64, 16), (128, 8), (1024, 1)]:
        a = np.cumprod(rng.uniform(0.6, 1.0, size=(R, gamma)), axis=1).astype(np.float32)
        sps = np.ones(R * (gamma + 1) + 1, np.float32)       # flat: every item is admitted
        ws = ds.Workspace(R, gamma, 8, 16, 0)
        ell, Bt, th = ds.schedule(torch.from_numpy(a).cuda(), torch.from_numpy(sps).cuda(), ws)
        ell_ref, Bt_ref, th_ref = oracle.schedule(a, sps)
        np.testing.assert_array_equal(ell.cpu().numpy(), ell_ref)
        assert int(Bt.item()) == Bt_ref == R * (gamma + 1) and float(th.item()) == th_ref
