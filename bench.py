"""Benchmark of one DSpark speculative step (draft -> confidence -> schedule -> verify).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path over one batch of
synthetic input (the seeded workloads module); every step draws with its own seed.
``value`` is draft+verify positions/s (B * gamma per step, summed over all ranks) with
the inputs resident in HBM; ``e2e`` is the same metric with the step's inputs copied in
from pinned host memory and the verified tokens copied back inside the timed region (the
next step's copies overlap the current step's kernels).

With N > 1 (torchrun, one rank per GPU) every rank runs an independent replica on its own
batch (the path shards by request; there is no data-path collective), timing is bracketed
by barriers and the slowest rank's time is used.

``--impl reference`` times the CPU oracle as it stands on this host's cores (rank 0 only),
each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "draft+verify positions/sec (B×γ) at V=151936, r=256; achieved HBM GB/s"


# DRAM bytes (read + write) per launch of the step's first kernel (the draft with the
# confidence head and the scheduler) at qwen3_4b_like, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel sources it was
# taken on: the sha1 of those files is checked at run time and the figure dropped (traffic
# null) once they change.
DRAFT_TRAFFIC = {"workload": "qwen3_4b_like", "bytes": 233_753_600,
                 "sources_sha1": "e02c8e9408c88bbb62432b5d7f855d1cbcb45ac2"}
DRAFT_SOURCES = ("draft.cu", "sm100_ptx.cuh", "common.cuh", "internal.h")
FIRST_KERNEL = ("draft_lanes_kernel via dspark_draft_confidence_schedule (bias contraction, "
                "sampling, confidence and schedule, all gamma positions)")
VERIFY_KERNELS = 5          # target statistics, decision, bias rows, final draw, finalize
FUSED_SCHEDULE_ITEMS = 4096  # the draft launch schedules up to this B*gamma itself


def launches_per_step(w) -> int:
    """Kernels of one benchmarked step: one launch drafts, scores confidence and (up to
    4096 items) schedules; larger batches schedule in a launch of their own; then the
    verification's kernels."""
    return 1 + (0 if w.B * w.gamma <= FUSED_SCHEDULE_ITEMS else 1) + VERIFY_KERNELS


def _draft_traffic(w):
    import hashlib
    if w.name != DRAFT_TRAFFIC["workload"]:
        return None
    h = hashlib.sha1()
    for f in DRAFT_SOURCES:
        with open(os.path.join(ROOT, "speculative_decoding_03_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return DRAFT_TRAFFIC["bytes"] if h.hexdigest() == DRAFT_TRAFFIC["sources_sha1"] else None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ----------------------------------------------------------------- algorithmic bytes

def draft_bytes(w) -> int:
    """Bytes the draft must move at least once: U, W2 (once per step), the W1 rows
    gathered, and the outputs (tokens, q, max, sum)."""
    return (w.B * w.gamma * w.V * 4 + w.r * w.V * 2 + w.B * w.gamma * w.r * 2 +
            w.B * w.gamma * 16)


def first_launch_bytes(w) -> int:
    """Bytes the step's first launch must move at least once: the draft's, the hidden
    states h, the confidence outputs c and a, and (scheduled in the same launch) ell."""
    return draft_bytes(w) + w.B * w.gamma * (w.H * 4 + 8) + w.H * 4 + w.B * 4


def step_bytes(w, n_out: np.ndarray, accept_len: np.ndarray, ell: np.ndarray) -> int:
    """Algorithmic bytes of one step: the draft's, h, the target rows needed up to each
    request's stop (n_out rows), and one U row for each request whose stop was a reject."""
    rejected = int(np.sum(accept_len < ell))
    return (draft_bytes(w) + w.B * w.gamma * w.H * 4 + int(np.sum(n_out)) * w.V * 4 +
            rejected * w.V * 4)


# ----------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"dspark_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower().startswith("active")})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------- CPU oracle

def oracle_sample_step(inp, seed: int, nthreads: int):
    """One oracle step (draft, confidence, schedule, verify) on already generated inputs
    (their requests as their own batch); returns the positions it drafted."""
    import oracle
    d = oracle.draft(inp.U, inp.W1, inp.W2, inp.anchor, seed, inp.requests, nthreads)
    _, a = oracle.confidence(inp.h, inp.anchor, d["tokens"], inp.W1, inp.w_c, float(inp.b_c))
    ell, _, _ = oracle.schedule(a.astype(np.float32), inp.sps)
    oracle.verify(inp.T, inp.U, inp.W1, inp.W2, inp.anchor, d["tokens"], ell, seed, inp.requests, nthreads)
    return len(inp.requests) * inp.w.gamma


def cpu_baseline(w, n_req: int):
    """The oracle as it stands on this host's cores, on a bounded request sample: one step
    of the first n_req requests with every core (OpenMP over requests), and one request on
    one thread.  Inputs are generated before the timed regions."""
    import oracle
    n = _cores()
    oracle.lib()
    n_req = max(1, min(w.B, n_req))
    inp = workloads.generate(w, requests=range(n_req))
    t0 = time.perf_counter()
    pos = oracle_sample_step(inp, w.seed, n)
    dt = time.perf_counter() - t0
    one = workloads.generate(w, requests=[0])
    t0 = time.perf_counter()
    pos1 = oracle_sample_step(one, w.seed, 1)
    dt1 = time.perf_counter() - t0
    return {"value": pos / dt, "unit": "positions/s", "cores": n, "kind": "oracle",
            "single_thread": {"value": pos1 / dt1, "unit": "positions/s", "cores": 1,
                              "sample": f"request 0 of {w.name}, one thread ({dt1:.2f} s)"},
            "sample": f"one full step (draft, confidence, schedule, verify) of the first {n_req} "
                      f"requests of {w.name} as their own batch, fp64, OpenMP over requests on "
                      f"{n} cores; {dt:.2f} s wall, input generation outside the timed region"}


# --------------------------------------------------------------------- reference arm

def run_reference(args, w):
    """The oracle as it stands, timed on this host's cores, rank 0 only.  Each step is a
    bounded sample of the workload (its first requests as their own batch, generated once
    before any timing; every step draws with its own seed): the first warm-up step runs
    the full sample and measures it, and the sample of the other steps is then sized so
    that the whole run (warm-up and timed steps) fits --ref-budget-s, down to one request
    per OpenMP thread (below that a step would not get shorter)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    n = _cores()
    oracle.lib()
    n_full = min(w.B, args.ref_requests)
    inp_full = workloads.generate(w, requests=range(n_full))
    t0 = time.perf_counter()
    oracle_sample_step(inp_full, w.seed, n)
    t_full = time.perf_counter() - t0
    # the oracle runs the requests in rounds of its OpenMP threads: size the sample in whole
    # rounds (at least one, so every thread still has a request)
    n_req = n_full
    remaining = (args.warmup - 1) + args.steps
    rounds_full = -(-n_full // max(1, n))
    if remaining > 0 and t_full * (1 + remaining) > args.ref_budget_s:
        per_step = max(0.0, args.ref_budget_s - t_full) / remaining
        rounds = max(1, int(per_step / (t_full / rounds_full)))
        n_req = min(n_full, rounds * max(1, n))
    inp = workloads.generate(w, requests=range(n_req)) if n_req != n_full else inp_full
    for i in range(1, args.warmup):
        oracle_sample_step(inp, w.seed + i, n)
    t0 = time.perf_counter()
    pos = 0
    for i in range(args.steps):
        pos += oracle_sample_step(inp, w.seed + args.warmup + i, n)
    dt = time.perf_counter() - t0
    value = pos / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "positions/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(w.describe(), sample_requests=n_req),
            "cpu_baseline": {"value": value, "unit": "positions/s", "cores": n, "kind": "oracle",
                             "sample": f"first {n_req} requests of {w.name} as their own batch per "
                                       f"step, generated once before timing, a new seed per step "
                                       f"(sized to a {args.ref_budget_s:.0f} s run; the full "
                                       f"{n_full}-request step took {t_full:.1f} s)"},
            "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- replicas (N > 1)

def replica_workload(w, rank: int):
    """Each rank is an independent replica with its own batch: the data seed shifts by rank."""
    return workloads.scaled(w, seed=w.seed + 1000 * rank) if rank else w


def max_over_ranks(t_ms: float, dist, device: str = "cpu") -> float:
    """The slowest rank's time (the whole job finishes with it); dist None: one process."""
    if dist is None:
        return t_ms
    import torch
    t = torch.tensor([t_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, w, ms_per_step: float) -> float:
    """Positions per second of all replicas together: every rank does B * gamma per step."""
    return world * w.B * w.gamma / (ms_per_step * 1e-3)


# ------------------------------------------------------------ the other workloads

def measure_workload(w, args, world: int, rank: int, local: int, barrier, dist=None):
    """The same step on another workload (the headline's procedure at a smaller step
    count): graph-replayed steps with inputs resident in HBM, the draft launch alone, the
    roofline of both, and the oracle's rate on a bounded sample of the same workload."""
    import torch
    import speculative_decoding_03_gb300 as ds
    wr = replica_workload(w, rank)
    inp = workloads.generate(wr)
    dev = ds.to_device(inp, f"cuda:{local}")
    step = ds.Step(dev, float(inp.b_c))
    stream = torch.cuda.current_stream()
    for i in range(3):
        step.run(seed=w.seed + i)
    n = max(3, min(args.steps, 50))
    n_ring = 8

    def time_graphs(gs):
        for g in gs:
            g.replay()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            gs[i % len(gs)].replay()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / n

    ms = time_graphs(step.capture([w.seed + 10 + j for j in range(n_ring)]))
    ms = max_over_ranks(ms, dist, f"cuda:{local}")
    res = step.results()
    first_ms = time_graphs(step.capture([w.seed + 20 + j for j in range(n_ring)], first_only=True))
    draft_ms = time_graphs(step.capture([w.seed + 30 + j for j in range(n_ring)], draft_only=True))
    # the verification alone (the last step's drafts and schedule), in a graph ring of its
    # own: its target rows and W2 stay warmer in L2 than after a draft
    x, d, ell = dev, step.draft_out, step.sched_out[0]
    vgs = []
    for j in range(n_ring):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ds.verify_packed(x["T"], x["U"], x["W1"], step.W2p, x["anchor"], d["tokens"], d["q_tok"],
                             d["row_max"], d["row_sumexp"], ell, w.seed + 40 + j, step.ws,
                             step.verify_out)
        vgs.append(g)
    verify_ms = time_graphs(vgs)
    peak, peak_kind = _peaks()
    fbytes, dbytes = first_launch_bytes(w), draft_bytes(w)
    sbytes = step_bytes(w, res["n_out"], res["accept_len"], res["ell"])
    out = {"config": w.describe(), "ms_per_step": ms, "value": whole_job_rate(world, w, ms),
           "unit": "positions/s",
           "roofline": {"bound": "hbm", "kernel": FIRST_KERNEL,
                        "achieved": fbytes / (first_ms * 1e-3) / 1e9, "peak": peak,
                        "peak_kind": peak_kind, "unit": "GB/s",
                        "frac": fbytes / (first_ms * 1e-3) / 1e9 / peak,
                        "algorithmic_bytes_per_launch": fbytes, "ms_per_launch": first_ms,
                        "draft_alone": {"ms_per_launch": draft_ms, "algorithmic_bytes": dbytes,
                                        "achieved": dbytes / (draft_ms * 1e-3) / 1e9}},
           "step_hbm": {"algorithmic_bytes": sbytes, "achieved": sbytes / (ms * 1e-3) / 1e9,
                        "unit": "GB/s", "frac": sbytes / (ms * 1e-3) / 1e9 / peak},
           "accept": {"mean_ell": float(np.mean(res["ell"])),
                      "mean_accept_len": float(np.mean(res["accept_len"])), "B_total": res["B_total"]},
           "verify_alone_ms": verify_ms,
           "gpu_launches_per_step": launches_per_step(w)}
    del step, dev, vgs
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, min(w.B, args.ref_requests))
    return out


# --------------------------------------------------------------------- our arm

def run_ours(args, w):
    import torch
    import speculative_decoding_03_gb300 as ds

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    ds.lib()
    # each rank is an independent replica with its own batch: shift the data seed by rank
    wr = replica_workload(w, rank)
    inp = workloads.generate(wr)
    dev = ds.to_device(inp, f"cuda:{local}")
    step = ds.Step(dev, float(inp.b_c))
    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        step.run(seed=w.seed + i)
    barrier()
    n_ring = 8
    if args.graph:
        # a ring of captured steps with distinct seeds: one host call per step
        graphs = step.capture([w.seed + args.warmup + j for j in range(n_ring)])
        for g in graphs:
            g.replay()
        barrier()
        run_step = lambda i: graphs[i % n_ring].replay()
    else:
        run_step = lambda i: step.run(seed=w.seed + args.warmup + i)

    # ---- timed region: K steps, inputs resident in HBM
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        ev0.record(stream)
        for i in range(args.steps):
            run_step(i)
        ev1.record(stream)
        barrier()
    t_ms = ev0.elapsed_time(ev1)
    t_ms = max_over_ranks(t_ms, dist, "cuda")
    ms_per_step = t_ms / args.steps
    res = step.results()

    # ---- dominant kernel: the step's first launch (draft, confidence and schedule), and
    # the draft call alone, each timed with events on its stream
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x = step.dev
    n_draft = max(3, min(args.steps, 50))

    def time_launch(run):
        barrier()
        ev_a.record(stream)
        for i in range(n_draft):
            run(i)
        ev_b.record(stream)
        barrier()
        return ev_a.elapsed_time(ev_b) / n_draft

    if args.graph:
        fgraphs = step.capture([w.seed + j for j in range(n_ring)], first_only=True)
        dgraphs = step.capture([w.seed + j for j in range(n_ring)], draft_only=True)
        for g in fgraphs + dgraphs:
            g.replay()
        first_ms = time_launch(lambda i: fgraphs[i % n_ring].replay())
        draft_ms = time_launch(lambda i: dgraphs[i % n_ring].replay())
    else:
        first_ms = time_launch(lambda i: step.first_launch(w.seed + i))
        draft_ms = time_launch(lambda i: ds.draft_packed(x["U"], x["W1"], step.W2p, x["anchor"],
                                                         w.seed + i, step.ws, step.draft_out))

    # ---- the variants of the step (greedy drafting, two-step capacity scheduler, fixed
    # threshold): whole steps in a graph ring, and the greedy draft launch alone
    variants = {}
    n_var = max(3, min(args.steps, 50))

    def time_graphs(gs, n):
        for g in gs:
            g.replay()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            gs[i % len(gs)].replay()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / n

    for sampling, scheduler in (("greedy", "theta"), ("gumbel", "async"), ("greedy", "threshold")):
        vs = ds.Step(dev, float(inp.b_c), ws=step.ws, W2p=step.W2p, sampling=sampling,
                     scheduler=scheduler, threshold=0.5)
        for i in range(3):
            vs.run(seed=w.seed + i, t=i)
        ms = time_graphs(vs.capture([w.seed + j for j in range(n_ring)]), n_var)
        vr = vs.results()
        entry = {"ms_per_step": ms, "value": whole_job_rate(world, w, ms),
                 "mean_ell": float(np.mean(vr["ell"])),
                 "mean_accept_len": float(np.mean(vr["accept_len"])), "B_total": vr["B_total"]}
        if sampling == "greedy" and scheduler == "theta":
            gd_ms = time_graphs(vs.capture([w.seed + j for j in range(n_ring)], draft_only=True), n_var)
            gd_ach = draft_bytes(w) / (gd_ms * 1e-3) / 1e9
            entry["draft"] = {"ms_per_launch": gd_ms, "achieved_gbs": gd_ach}
        variants[f"{sampling}+{scheduler}"] = entry
        del vs
    # the RNN head (its own weights; the step projects the hidden states first)
    W_rnn, b_rnn = workloads.gen_rnn_weights(wr)
    ds.rnn_to_device(W_rnn, b_rnn, dev, f"cuda:{local}")
    vs = ds.Step(dev, float(inp.b_c), ws=step.ws, W2p=step.W2p, head="rnn")
    for i in range(3):
        vs.run(seed=w.seed + i)
    ms = time_graphs(vs.capture([w.seed + j for j in range(n_ring)]), n_var)
    vr = vs.results()
    rd_ms = time_graphs(vs.capture([w.seed + j for j in range(n_ring)], draft_only=True), n_var)
    # the projection and the RNN draft kernel alone, each in its own graphs
    pg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pg):
        for i in range(10):
            ds.rnn_project(x["h"], dev["W_rnn"], dev["b_rnn"], vs.hp)
    proj_ms = time_graphs([pg], max(1, n_var // 10)) / 10
    dgs = []
    for j in range(n_ring):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ds.draft_rnn(x["U"], x["W1"], step.W2p, vs.Wrec, vs.hp, x["anchor"], w.seed + j, step.ws,
                         packed=True, out=vs.draft_out)
        dgs.append(g)
    dk_ms = time_graphs(dgs, n_var)
    variants["gumbel+theta+rnn_head"] = {
        "ms_per_step": ms, "value": whole_job_rate(world, w, ms),
        "mean_ell": float(np.mean(vr["ell"])), "mean_accept_len": float(np.mean(vr["accept_len"])),
        "B_total": vr["B_total"],
        "draft": {"ms_per_call": rd_ms, "project_ms": proj_ms, "draft_kernel_ms": dk_ms}}
    del vs

    # ---- per-call breakdown (warm, eager, events between the calls on one stream); the
    # step runs confidence and schedule as one launch, timed here both ways
    n_bd = max(3, min(args.steps, 20))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    acc = [0.0] * 6
    d_out, c_out, s_out, v_out = step.draft_out, step.conf_out, step.sched_out, step.verify_out
    for i in range(n_bd):
        sd = w.seed + 500 + i
        evs[0].record(stream)
        ds.draft_packed(x["U"], x["W1"], step.W2p, x["anchor"], sd, step.ws, d_out)
        evs[1].record(stream)
        ds.confidence(x["h"], x["anchor"], d_out["tokens"], x["W1"], x["w_c"], step.b_c, step.ws, c_out)
        evs[2].record(stream)
        ds.schedule(c_out[1], x["sps"], step.ws, s_out)
        evs[3].record(stream)
        ds.confidence_schedule(x["h"], x["anchor"], d_out["tokens"], x["W1"], x["w_c"], step.b_c,
                               x["sps"], step.ws, c_out, s_out)
        evs[4].record(stream)
        ds.verify_packed(x["T"], x["U"], x["W1"], step.W2p, x["anchor"], d_out["tokens"],
                         d_out["q_tok"], d_out["row_max"], d_out["row_sumexp"], s_out[0], sd,
                         step.ws, v_out)
        evs[5].record(stream)
        step.first_launch(sd)
        evs[6].record(stream)
        torch.cuda.synchronize()
        for j in range(6):
            acc[j] += evs[j].elapsed_time(evs[j + 1])
    breakdown = {k: acc[j] / n_bd for j, k in enumerate(
        ("draft_ms", "confidence_ms", "schedule_ms", "confidence_schedule_ms", "verify_ms",
         "draft_confidence_schedule_ms"))}

    # ---- end to end through the public API with pinned host buffers
    hin, hout = step.pinned_host_buffers()
    for k in step.STEP_INPUTS:
        hin[k].copy_(x[k].cpu())
    # (the pipeline overlaps step i + 1's host->device copies with step i's kernels; every
    # step still copies its inputs from pinned host memory and its tokens back)
    n_e2e = max(3, min(args.steps, 20))
    pipe = step.pipeline()
    pipe.run([w.seed, w.seed + 1], [hin, hin], [hout, hout])
    torch.cuda.current_stream().synchronize()
    barrier()
    t0 = time.perf_counter()
    pipe.run([w.seed + i for i in range(n_e2e)], [hin] * n_e2e, [hout] * n_e2e)
    torch.cuda.current_stream().synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e
    # bytes per step: the copied inputs, the target rows each step fetched (its
    # sum_b (l_b + 1), replayed here on the same inputs and seeds) and the tokens back
    rows = []
    for i in range(n_e2e):
        step.first_launch(w.seed + i)
        rows.append(int(step.sched_out[1].item()))
    h2d, d2h = step.step_bytes(B_total=float(np.mean(rows)))

    # the other workloads, each measured the same way on every replica (barriers included)
    per_workload = {}
    if args.per_workload:
        for other in workloads.WORKLOADS:
            if other.name != w.name:
                per_workload[other.name] = measure_workload(other, args, world, rank, local, barrier, dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = _peaks()
    fbytes, dbytes = first_launch_bytes(w), draft_bytes(w)
    achieved = fbytes / (first_ms * 1e-3) / 1e9
    sbytes = step_bytes(w, res["n_out"], res["accept_len"], res["ell"])
    line = {
        "metric": METRIC,
        "value": whole_job_rate(world, w, ms_per_step),
        "unit": "positions/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(w.describe(), weights="bf16", logits="fp32",
                       l2="inputs larger than L2 (U+T alone %.0f MB per step)" %
                          ((w.B * w.gamma * w.V + w.B * (w.gamma + 1) * w.V) * 4 / 1e6),
                       parallelism=f"replicas x{world}",
                       launch="cuda graph ring of 8 seeds" if args.graph else "eager"),
        "roofline": {"bound": "hbm", "kernel": FIRST_KERNEL,
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _draft_traffic(w),
                     "algorithmic_bytes_per_launch": fbytes, "ms_per_launch": first_ms,
                     "draft_alone": {"ms_per_launch": draft_ms, "algorithmic_bytes": dbytes,
                                     "achieved": dbytes / (draft_ms * 1e-3) / 1e9}},
        "step_hbm": {"algorithmic_bytes": sbytes, "achieved": sbytes / (ms_per_step * 1e-3) / 1e9,
                     "unit": "GB/s", "frac": sbytes / (ms_per_step * 1e-3) / 1e9 / peak},
        "accept": {"mean_ell": float(np.mean(res["ell"])), "mean_accept_len": float(np.mean(res["accept_len"])),
                   "B_total": res["B_total"], "theta": res["theta"]},
        "breakdown": breakdown,
        "variants": variants,
        "e2e": {"value": whole_job_rate(world, w, e2e_s * 1e3), "unit": "positions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, min(w.B, args.ref_requests))
    if per_workload:
        line["per_workload"] = per_workload
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="qwen3_4b_like", choices=[w.name for w in workloads.WORKLOADS])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-requests", type=int, default=32)
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="wall-time budget of the reference arm (its per-step sample is sized to it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", dest="per_workload", action="store_false",
                    help="skip the other workloads' block")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch every call from Python instead of replaying captured steps")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    w = workloads.get(args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
