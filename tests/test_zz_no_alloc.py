"""The allocation-free draft entry point (dspark_draft_noalloc) against dspark_draft.

dspark_draft_noalloc serves callers that cannot allocate device memory when they draft
(a serving loop whose memory is all held by its own pool, a plugin that only receives its
input and output buffers); its scratch is a fixed array inside the library instead of a
caller workspace.  This test calls it through the C ABI twice in a row and checks each
result against dspark_draft on the same inputs and seed, with the tolerances of the other
parity tests: identical token ids, probabilities within 1e-5 relative.  It also checks
that batches beyond the array's limit are refused.

The file name sorts last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
ds = pytest.importorskip("speculative_decoding_03_gb300")

RTOL = 1e-5


def _noalloc(dev, w, seed):
    B, gamma, V = dev["U"].shape
    r = dev["W1"].shape[1]
    out = dict(tokens=torch.full((B, gamma), -7, dtype=torch.int32, device="cuda"),
               q_tok=torch.zeros((B, gamma), dtype=torch.float32, device="cuda"),
               row_max=torch.zeros((B, gamma), dtype=torch.float32, device="cuda"),
               row_sumexp=torch.zeros((B, gamma), dtype=torch.float32, device="cuda"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = ds.lib().dspark_draft_noalloc(
        dev["U"].data_ptr(), dev["W1"].data_ptr(), dev["W2"].data_ptr(), dev["anchor"].data_ptr(),
        B, gamma, V, r, ctypes.c_uint64(seed), out["tokens"].data_ptr(), out["q_tok"].data_ptr(),
        out["row_max"].data_ptr(), out["row_sumexp"].data_ptr(), stream)
    assert rc == 0, ds.STATUS.get(rc, rc)
    return out


@pytest.mark.parametrize("name", ["qwen_small", "two_chunks"])
def test_noalloc_draft_matches_workspace_draft_twice(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if name == "qwen_small":
        w = workloads.scaled(workloads.get("qwen3_4b_like"), B=32, gamma=7, V=20008, r=256, H=32)
    else:
        w = workloads.scaled(workloads.get("production"), B=40, gamma=5, V=2056, r=128, H=16)
    inp = workloads.generate(w, with_T=False)
    dev = ds.to_device(inp, "cuda")
    ws = ds.Workspace(w.B, w.gamma, w.V, w.r, w.H)
    for seed in (w.seed, w.seed + 12345):            # two calls in a row
        got = {k: v.cpu().numpy() for k, v in _noalloc(dev, w, seed).items()}
        ref = {k: v.cpu().numpy() for k, v in
               ds.draft(dev["U"], dev["W1"], dev["W2"], dev["anchor"], seed, ws).items()}
        np.testing.assert_array_equal(got["tokens"], ref["tokens"])
        for key in ("q_tok", "row_max", "row_sumexp"):
            np.testing.assert_allclose(got[key], ref[key], rtol=RTOL, err_msg=key)
    assert ws.status() == 0


def test_noalloc_refuses_batches_beyond_its_limit():
    L = ds.lib()
    fake = 0x10000000
    args = lambda B, gamma: (fake, fake, fake, fake, B, gamma, 1000, 16, ctypes.c_uint64(0),
                             fake, fake, fake, fake, None)
    assert L.dspark_draft_noalloc(*args(257, 4)) == 2          # DSPARK_ERR_UNSUPPORTED
    assert L.dspark_draft_noalloc(*args(4, 33)) == 2
    assert L.dspark_draft_noalloc(*args(0, 4)) == 1            # DSPARK_ERR_INVALID_ARG
