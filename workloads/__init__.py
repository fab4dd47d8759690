"""Seeded synthetic inputs for the DSpark per-step hot path.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It only draws random numbers and lays them out; it holds none of the
method's arithmetic (no softmax, no bias, no sampling, no scheduling).

What the inputs stand for (DSpark pages, "DSpark: Confidence-Scheduled
Speculative Decoding with Semi-Autoregressive Generation" as summarised on
billytse.dev, section 3.1 "Parallel backbone" and section 3.3 "Markov head"):

* ``U``  [B, gamma, V] fp32 -- the parallel backbone's base logits U_k;
* ``T``  [B, gamma+1, V] fp32 -- the target model's logits for the gamma draft
  positions plus one bonus row (the target's extra token when every verified
  position is accepted);
* ``W1`` [V, r] and ``W2`` [r, V] bf16 (stored as uint16 bit patterns) -- the
  low-rank Markov head, bias(prev, .) = W1[prev] @ W2, rank r;
* ``h``  [B, gamma, H] fp32 -- the backbone's per-position hidden states;
* ``w_c`` [H + r] fp32 and ``b_c`` -- the confidence head (one linear layer on
  [h_k ; W1[prev]] followed by a sigmoid);
* ``anchor`` [B] int32 -- the last committed token of each request;
* ``sps`` [R*(gamma+1) + 1] fp32 -- the profiled steps-per-second curve SPS(B)
  indexed by the integer token-batch size B;
* ``W_rnn`` [2r + H, 3r] bf16 and ``b_rnn`` [3r] fp32 (``gen_rnn_weights``) -- the RNN
  head's one linear layer on [state ; previous-token embedding ; hidden state], its
  output columns in three blocks (gate, candidate, output).

The pages measure on live traffic and on datasets that are not available here;
these seeded draws stand in for them.  Every request's rows come from their own
numpy ``default_rng([seed, stream, b])`` so that any subset of requests can be
regenerated on its own (the oracle checks sampled requests at full size).
"""
from __future__ import annotations

import dataclasses
import os
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

# random-stream identifiers, one per tensor
_S_U, _S_T, _S_W1, _S_W2, _S_H, _S_WC, _S_ANCHOR, _S_WRNN = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, value distributions and the SPS curve."""

    name: str
    B: int                      # requests R = B
    gamma: int                  # draft block length
    V: int                      # vocabulary size
    r: int                      # Markov rank
    H: int                      # drafter hidden size
    seed: int                   # data seed; the sampling seed defaults to it too
    u_std: float                # std of the base logits U
    spike_p: float              # Bernoulli probability of a spike per (b, k, v)
    spike_amp: float            # spike height added to U
    noise_std: Callable[[int], float]   # target perturbation std at position k (1-based)
    sps_fn: Callable[[np.ndarray], np.ndarray]  # SPS(B) for integer B
    w_std: float = 0.02         # std of W1, W2 before bf16 rounding
    b_c: float = 1.0            # confidence-head bias

    @property
    def sps_len(self) -> int:
        return self.B * (self.gamma + 1) + 1

    def describe(self) -> Dict[str, object]:
        return {"workload": self.name, "B": self.B, "gamma": self.gamma, "V": self.V,
                "r": self.r, "H": self.H, "seed": self.seed}


def _pw_linear(knots: Sequence[tuple]) -> Callable[[np.ndarray], np.ndarray]:
    xs = np.array([k[0] for k in knots], dtype=np.float64)
    ys = np.array([k[1] for k in knots], dtype=np.float64)

    def f(b: np.ndarray) -> np.ndarray:
        return np.interp(b.astype(np.float64), xs, ys)
    return f


_PROD_KNOTS = [(0, 1.00), (256, 0.97), (512, 0.90), (768, 0.80), (1024, 0.72),
               (1025, 0.66), (1536, 0.52), (2048, 0.40)]

WORKLOADS: List[Workload] = [
    Workload("tiny", B=4, gamma=4, V=1000, r=16, H=64, seed=0,
             u_std=2.0, spike_p=0.0, spike_amp=0.0,
             noise_std=lambda k: 1.0,
             sps_fn=lambda b: 1.0 / (1.0 + 0.01 * b)),
    Workload("qwen3_4b_like", B=32, gamma=7, V=151936, r=256, H=2560, seed=1,
             u_std=3.0, spike_p=0.01, spike_amp=8.0,
             noise_std=lambda k: 1.0,
             sps_fn=lambda b: 1.0 / (1.0 + 0.005 * np.maximum(0, b - 64))),
    Workload("production", B=256, gamma=5, V=129280, r=256, H=4096, seed=2,
             u_std=3.0, spike_p=0.01, spike_amp=8.0,
             noise_std=lambda k: 1.5,
             sps_fn=_pw_linear(_PROD_KNOTS)),
    Workload("long_block", B=128, gamma=15, V=151936, r=256, H=2560, seed=3,
             u_std=3.0, spike_p=0.01, spike_amp=8.0,
             noise_std=lambda k: 0.5 + 1.5 * (k - 1) / 14.0,
             sps_fn=_pw_linear(_PROD_KNOTS)),
    Workload("scheduler_stress", B=1024, gamma=16, V=32768, r=128, H=2048, seed=4,
             u_std=3.0, spike_p=0.01, spike_amp=8.0,
             noise_std=lambda k: 1.0,
             sps_fn=lambda b: 1.0 / (1.0 + np.maximum(0, b - 512) / 512.0)),
]

BY_NAME: Dict[str, Workload] = {w.name: w for w in WORKLOADS}


def get(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    return BY_NAME[name_or_index]


def scaled(w: Workload, **kw) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **kw)


def _rng(seed: int, stream: int, *idx: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream, *idx])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even) and return the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _logit_rows(rng: np.random.Generator, rows: int, V: int, w: Workload) -> np.ndarray:
    x = rng.standard_normal((rows, V), dtype=np.float32)
    x *= np.float32(w.u_std)
    if w.spike_p > 0.0:
        spikes = rng.random((rows, V), dtype=np.float32) < np.float32(w.spike_p)
        x += spikes.astype(np.float32) * np.float32(w.spike_amp)
    return x


def gen_U_T(w: Workload, b: int, with_T: bool = True):
    """Base logits U[b] (gamma x V) and target logits T[b] ((gamma+1) x V) of request b."""
    U = _logit_rows(_rng(w.seed, _S_U, b), w.gamma, w.V, w)
    if not with_T:
        return U, None
    rng = _rng(w.seed, _S_T, b)
    T = np.empty((w.gamma + 1, w.V), dtype=np.float32)
    for k in range(1, w.gamma + 1):
        T[k - 1] = U[k - 1] + rng.standard_normal(w.V, dtype=np.float32) * np.float32(w.noise_std(k))
    T[w.gamma] = _logit_rows(rng, 1, w.V, w)[0]
    return U, T


def gen_weights(w: Workload):
    """W1 [V, r] and W2 [r, V] as bf16 bit patterns (uint16), w_c [H+r] fp32, b_c."""
    W1 = f32_to_bf16_bits(_rng(w.seed, _S_W1).standard_normal((w.V, w.r), dtype=np.float32)
                          * np.float32(w.w_std))
    W2 = f32_to_bf16_bits(_rng(w.seed, _S_W2).standard_normal((w.r, w.V), dtype=np.float32)
                          * np.float32(w.w_std))
    w_c = (_rng(w.seed, _S_WC).standard_normal(w.H + w.r) / np.sqrt(w.H + w.r)).astype(np.float32)
    return W1, W2, w_c, np.float32(w.b_c)


def gen_rnn_weights(w: Workload):
    """W_rnn [2r + H, 3r] bf16 bits and b_rnn [3r] fp32 of the RNN head.

    W_rnn ~ N(0, 1/(r + H)) so that a pre-activation, a sum over r state entries in
    (-1, 1), r small embedding entries and H unit-variance hidden entries, is of order
    one; the gate block's bias is +1 (the state is mostly kept), the other biases 0."""
    rng = _rng(w.seed, _S_WRNN)
    W = rng.standard_normal((2 * w.r + w.H, 3 * w.r), dtype=np.float32) * np.float32(1.0 / np.sqrt(w.r + w.H))
    b = np.zeros(3 * w.r, dtype=np.float32)
    b[:w.r] = 1.0
    return f32_to_bf16_bits(W), b


def gen_h(w: Workload, b: int) -> np.ndarray:
    return _rng(w.seed, _S_H, b).standard_normal((w.gamma, w.H), dtype=np.float32)


def gen_anchor(w: Workload) -> np.ndarray:
    return _rng(w.seed, _S_ANCHOR).integers(0, w.V, size=w.B, dtype=np.int64).astype(np.int32)


def gen_sps(w: Workload) -> np.ndarray:
    return np.asarray(w.sps_fn(np.arange(w.sps_len)), dtype=np.float32)


@dataclasses.dataclass
class Inputs:
    w: Workload
    U: np.ndarray
    T: Optional[np.ndarray]
    W1: np.ndarray
    W2: np.ndarray
    h: np.ndarray
    w_c: np.ndarray
    b_c: np.float32
    anchor: np.ndarray
    sps: np.ndarray
    requests: np.ndarray     # which request indices these rows belong to


def generate(w: Workload, requests: Optional[Sequence[int]] = None, with_T: bool = True) -> Inputs:
    """All inputs of ``w``; with ``requests`` only those requests' per-request rows.

    Weights, the SPS table and the anchors are always generated in full (anchors are
    then restricted to ``requests``)."""
    reqs = np.arange(w.B) if requests is None else np.asarray(list(requests), dtype=np.int64)
    n = len(reqs)
    U = np.empty((n, w.gamma, w.V), dtype=np.float32)
    T = np.empty((n, w.gamma + 1, w.V), dtype=np.float32) if with_T else None
    h = np.empty((n, w.gamma, w.H), dtype=np.float32)

    def one(i: int) -> None:
        b = int(reqs[i])
        u, t = gen_U_T(w, b, with_T)
        U[i] = u
        if with_T:
            T[i] = t
        h[i] = gen_h(w, b)

    # every request draws from its own generator, so the rows do not depend on the order
    # (or the thread) they are made in; numpy releases the GIL while it fills large arrays
    if n * w.gamma * w.V >= (1 << 24):
        import concurrent.futures as cf
        try:
            workers = max(1, min(16, len(os.sched_getaffinity(0))))
        except AttributeError:  # pragma: no cover
            workers = max(1, min(16, os.cpu_count() or 1))
        with cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(n)))
    else:
        for i in range(n):
            one(i)
    W1, W2, w_c, b_c = gen_weights(w)
    anchor = gen_anchor(w)[reqs]
    return Inputs(w, U, T, W1, W2, h, w_c, b_c, anchor, gen_sps(w), reqs)
