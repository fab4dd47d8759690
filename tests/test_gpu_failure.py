"""Failure detection on the GPU without a GPU fault: a bounded wait of the draft kernels is
made to run out, and the library must report it and stay usable.

The draft kernels bound every wait (their shared-memory pipelines, their grid barriers).  The
library's testing hook shortens the bound to about a millisecond and moves the grid
barrier's target out of reach, so the first position's barrier cannot complete: every CTA
gives up, records DSPARK_ERR_TIMEOUT, drains its copies and MMAs, frees its tensor memory
and returns.  The host then reads the status, restores the production setting, and a
normal draft on the same workspace must succeed and match the oracle.
"""
import numpy as np
import pytest

import oracle
import workloads
from _parity import draft_rows, draft_stats

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
ds = pytest.importorskip("speculative_decoding_03_gb300")

TIMEOUT = 4          # DSPARK_ERR_TIMEOUT


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name,greedy", [("qwen_small", False), ("wide_batch", True)])
def test_draft_wait_runs_out_and_the_next_call_succeeds(name, greedy):
    _need_gpu()
    w = {"qwen_small": workloads.scaled(workloads.get("qwen3_4b_like"), B=5, gamma=3, V=904, r=64, H=32),
         "wide_batch": workloads.scaled(workloads.get("scheduler_stress"), B=300, gamma=2, V=520, r=128, H=8)}[name]
    inp = workloads.generate(w, with_T=False)
    dev = ds.to_device(inp)
    ws = ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)
    call = (lambda: ds.draft_greedy(dev["U"], dev["W1"], dev["W2"], dev["anchor"], ws)) if greedy else \
        (lambda: ds.draft(dev["U"], dev["W1"], dev["W2"], dev["anchor"], w.seed, ws))
    try:
        ds.testing_set_wait_limit(2_000_000, unreachable_barrier=True)   # ~1 ms at 2 GHz
        call()
        assert ws.status() == TIMEOUT
    finally:
        ds.testing_set_wait_limit()
    assert ws.status() == 0                                 # read and cleared
    got = {k: v.cpu().numpy() for k, v in call().items()}
    assert ws.status() == 0
    ref = oracle.draft_greedy(inp.U, inp.W1, inp.W2, inp.anchor) if greedy else \
        oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, w.seed)
    _, same = draft_rows(got["tokens"], ref["tokens"], ref["gap"], name)
    draft_stats(got, ref, same, keys=("row_max", "row_sumexp") if greedy else
                ("q_tok", "row_max", "row_sumexp"), label=name)


def test_rnn_draft_wait_runs_out_and_the_next_call_succeeds():
    """The RNN head's draft kernel has two exchanges per position (the recurrence CTAs'
    arrival count and the grid barrier); with both targets out of reach every wait runs out,
    the call reports DSPARK_ERR_TIMEOUT, and the next call matches the oracle."""
    _need_gpu()
    w = workloads.scaled(workloads.get("qwen3_4b_like"), B=5, gamma=3, V=904, r=64, H=32)
    inp = workloads.generate(w, with_T=False)
    W_rnn, b_rnn = workloads.gen_rnn_weights(w)
    dev = ds.rnn_to_device(W_rnn, b_rnn, ds.to_device(inp))
    ws = ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)
    hp = torch.from_numpy(np.ascontiguousarray(oracle.rnn_project(inp.h, W_rnn, b_rnn),
                                               dtype=np.float32)).cuda()
    Wrec = ds.rnn_pack(dev["W_rnn"], w.r)
    call = lambda: ds.draft_rnn(dev["U"], dev["W1"], dev["W2"], Wrec, hp, dev["anchor"], w.seed, ws)
    try:
        ds.testing_set_wait_limit(2_000_000, unreachable_barrier=True)
        call()
        assert ws.status() == TIMEOUT
    finally:
        ds.testing_set_wait_limit()
    assert ws.status() == 0
    got = {k: v.cpu().numpy() for k, v in call().items()}
    assert ws.status() == 0
    ref = oracle.draft_rnn(inp.U, inp.h, inp.W1, inp.W2, W_rnn, b_rnn, inp.anchor, w.seed)
    _, same = draft_rows(got["tokens"], ref["tokens"], ref["gap"], "rnn")
    draft_stats(got, ref, same, keys=("q_tok", "row_max", "row_sumexp"), label="rnn")
