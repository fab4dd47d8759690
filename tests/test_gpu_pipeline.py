"""The host pipeline (next step's host->device copies overlapped with the current step)
gives, step by step, exactly the tokens of the same steps run one at a time."""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
ds = pytest.importorskip("speculative_decoding_03_gb300")


def test_pipeline_matches_steps_run_one_at_a_time():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = workloads.scaled(workloads.get("qwen3_4b_like"), B=8, gamma=4, V=3000, r=64, H=32)
    base = workloads.generate(w)
    seeds = [11, 12, 13]
    # three steps' inputs: the base batch and two perturbed ones (same weights)
    per_step = []
    for i in range(3):
        rng = np.random.default_rng(100 + i)
        per_step.append({
            "U": (base.U + (rng.normal(0, 0.5, base.U.shape) if i else 0)).astype(np.float32),
            "T": (base.T + (rng.normal(0, 0.5, base.T.shape) if i else 0)).astype(np.float32),
            "h": (base.h + (rng.normal(0, 0.1, base.h.shape) if i else 0)).astype(np.float32),
            "anchor": (rng.permutation(base.anchor) if i else base.anchor).astype(np.int32),
        })
    # reference: each step on its own, inputs resident
    ref = []
    for x, sd in zip(per_step, seeds):
        dev = ds.to_device(base)
        for k, v in x.items():
            dev[k] = torch.from_numpy(v).cuda()
        ref.append(ds.Step(dev, float(base.b_c)).run(seed=sd).results())
    # pipeline: one Step, every step's inputs copied from pinned host buffers
    step = ds.Step(ds.to_device(base), float(base.b_c))
    hins, houts = [], []
    for x in per_step:
        hin, hout = step.pinned_host_buffers()
        for k in step.STEP_INPUTS:
            hin[k].copy_(torch.from_numpy(x[k]))
        hins.append(hin)
        houts.append(hout)
    step.pipeline().run(seeds, hins, houts)
    torch.cuda.synchronize()
    assert step.ws.status() == 0
    for i in range(3):
        for k in step.STEP_OUTPUTS:
            np.testing.assert_array_equal(houts[i][k].numpy(), ref[i][k], err_msg=f"step {i} {k}")
