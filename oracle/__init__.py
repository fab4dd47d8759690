"""CPU oracle of the DSpark per-step hot path (ctypes wrapper around dspark_oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import this package.  The
CUDA library never calls it and shares no code with it.

Every function computes in fp64 from the fp32 / bf16 inputs; see dspark_oracle.c for
the passages each part follows and for the readings taken where the pages are silent.
The parity pins of each function are the ``tests/test_oracle_*.py`` tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")

# the command the build step runs too; -ffp-contract=off keeps every product and sum a
# separately rounded IEEE operation (no fused multiply-add), on x86 and on Arm alike
GCC_CMD = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", _OUT, _SRC, "-lm"]

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_OUT), exist_ok=True)
        subprocess.run(GCC_CMD, check=True)
    return _OUT


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, u64, f32 = ctypes.c_int, ctypes.c_uint64, ctypes.c_float
        L.dso_philox4x32.argtypes = [P, u64, ctypes.c_int, P]
        L.dso_philox4x32.restype = None
        L.dso_draw.argtypes = [u64, i32, i32, i32, i32]
        L.dso_draw.restype = ctypes.c_uint32
        L.dso_u01.argtypes = [ctypes.c_uint32]
        L.dso_u01.restype = ctypes.c_double
        L.dso_one_minus_u01.argtypes = [ctypes.c_uint32]
        L.dso_one_minus_u01.restype = ctypes.c_double
        L.dso_gumbel.argtypes = [ctypes.c_uint32]
        L.dso_gumbel.restype = ctypes.c_double
        L.dso_draft.argtypes = [P, P, P, P, P, i32, i32, i32, i32, u64, P, P, P, P, P, i32]
        L.dso_draft.restype = i32
        L.dso_markov_bias.argtypes = [P, P, P, i32, i32, i32, P]
        L.dso_markov_bias.restype = i32
        L.dso_confidence.argtypes = [P, P, P, P, P, f32, i32, i32, i32, i32, i32, P, P]
        L.dso_confidence.restype = i32
        L.dso_schedule.argtypes = [P, i32, i32, P, i32, P, P, P]
        L.dso_schedule.restype = i32
        L.dso_verify.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, u64,
                                 P, P, P, P, P, P, i32]
        L.dso_verify.restype = i32
        L.dso_draft_greedy.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, P, P, P, i32]
        L.dso_draft_greedy.restype = i32
        L.dso_verify_greedy.argtypes = [P, P, P, P, i32, i32, i32, u64, P, P, P, P, P, P, i32]
        L.dso_verify_greedy.restype = i32
        L.dso_schedule_async.argtypes = [P, i32, i32, P, i32, i32, P, P, P, P]
        L.dso_schedule_async.restype = i32
        L.dso_schedule_threshold.argtypes = [P, i32, i32, f32, P, P]
        L.dso_schedule_threshold.restype = i32
        L.dso_rnn_project.argtypes = [P, P, P, i32, i32, i32, P]
        L.dso_rnn_project.restype = i32
        L.dso_draft_rnn.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, u64, i32,
                                    P, P, P, P, P, P, P, i32]
        L.dso_draft_rnn.restype = i32
        L.dso_verify_rnn.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, u64,
                                     P, P, P, P, P, P, i32]
        L.dso_verify_rnn.restype = i32
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


# ------------------------------------------------------------------------ random numbers

PHILOX_ROUNDS = 7   # the generator every draw uses: Philox4x32-7


def philox4x32(counter: Sequence[int], seed: int, rounds: int = PHILOX_ROUNDS) -> np.ndarray:
    ctr = _c(counter, np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().dso_philox4x32(_p(ctr), ctypes.c_uint64(seed), int(rounds), _p(out))
    return out


def draw(seed: int, b: int, k: int, v: int, stream: int) -> int:
    return int(lib().dso_draw(seed, b, k, v, stream))


def u01(x: int) -> float:
    return float(lib().dso_u01(x))


def one_minus_u01(x: int) -> float:
    return float(lib().dso_one_minus_u01(x))


def gumbel(x: int) -> float:
    return float(lib().dso_gumbel(x))


# ------------------------------------------------------------------------ the four calls

def draft(U, W1, W2, anchor, seed: int, req_ids: Optional[Sequence[int]] = None,
          nthreads: Optional[int] = None):
    """Semi-autoregressive draft of every request in ``U`` ([n, gamma, V]).

    Returns dict(tokens, q_tok, row_max, row_sumexp, gap) with [n, gamma] arrays."""
    U = _c(U, np.float32)
    n, gamma, V = U.shape
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    r = W1.shape[1]
    assert W1.shape == (V, r) and W2.shape == (r, V)
    anchor = _c(anchor, np.int32)
    ids = _c(np.arange(n) if req_ids is None else req_ids, np.int32)
    out = {k: np.zeros((n, gamma), dtype=np.float64) for k in ("q_tok", "row_max", "row_sumexp", "gap")}
    tokens = np.zeros((n, gamma), dtype=np.int32)
    rc = lib().dso_draft(_p(U), _p(W1), _p(W2), _p(anchor), _p(ids), n, gamma, V, r,
                         ctypes.c_uint64(seed), _p(tokens), _p(out["q_tok"]), _p(out["row_max"]),
                         _p(out["row_sumexp"]), _p(out["gap"]), nthreads or default_threads())
    _check(rc, "draft")
    out["tokens"] = tokens
    return out


def markov_bias(W1, W2, prev):
    """bias [n, V] = W1[prev] @ W2 in fp64 (prev = -1 gives a zero row)."""
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    V, r = W1.shape
    prev = _c(prev, np.int32)
    out = np.zeros((len(prev), V), dtype=np.float64)
    _check(lib().dso_markov_bias(_p(W1), _p(W2), _p(prev), len(prev), V, r, _p(out)), "markov_bias")
    return out


def confidence(h, anchor, tokens, W1, w_c, b_c: float):
    """Confidence c [n, gamma] and survival a [n, gamma]."""
    h = _c(h, np.float32)
    n, gamma, H = h.shape
    W1 = _c(W1, np.uint16)
    V, r = W1.shape
    w_c = _c(w_c, np.float32)
    assert w_c.shape == (H + r,)
    c = np.zeros((n, gamma), dtype=np.float64)
    a = np.zeros((n, gamma), dtype=np.float64)
    rc = lib().dso_confidence(_p(h), _p(_c(anchor, np.int32)), _p(_c(tokens, np.int32)), _p(W1),
                              _p(w_c), ctypes.c_float(b_c), n, gamma, H, r, V, _p(c), _p(a))
    _check(rc, "confidence")
    return c, a


def schedule(a, sps):
    """Prefix scheduler on survival a [R, gamma] (fp32) and SPS table sps (fp32).

    Returns (ell [R] int32, B_total, Theta)."""
    a = _c(a, np.float32)
    R, gamma = a.shape
    sps = _c(sps, np.float32)
    ell = np.zeros(R, dtype=np.int32)
    Bt = np.zeros(1, dtype=np.int32)
    th = np.zeros(1, dtype=np.float64)
    rc = lib().dso_schedule(_p(a), R, gamma, _p(sps), len(sps), _p(ell), _p(Bt), _p(th))
    _check(rc, "schedule")
    return ell, int(Bt[0]), float(th[0])


def verify(T, U, W1, W2, anchor, tokens, ell, seed: int, req_ids: Optional[Sequence[int]] = None,
           nthreads: Optional[int] = None):
    """Rejection-sampling verification of ``tokens`` with verified lengths ``ell``.

    Returns dict(accept_len [n], out_tokens [n, gamma+1], n_out [n], band [n, gamma],
    gap [n], fallback [n])."""
    T = _c(T, np.float32)
    U = _c(U, np.float32)
    n, gamma, V = U.shape
    assert T.shape == (n, gamma + 1, V)
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    r = W1.shape[1]
    ids = _c(np.arange(n) if req_ids is None else req_ids, np.int32)
    res = dict(accept_len=np.zeros(n, np.int32), out_tokens=np.zeros((n, gamma + 1), np.int32),
               n_out=np.zeros(n, np.int32), band=np.zeros((n, gamma), np.float64),
               gap=np.zeros(n, np.float64), fallback=np.zeros(n, np.int32))
    rc = lib().dso_verify(_p(T), _p(U), _p(W1), _p(W2), _p(_c(anchor, np.int32)),
                          _p(_c(tokens, np.int32)), _p(_c(ell, np.int32)), _p(ids), n, gamma, V, r,
                          ctypes.c_uint64(seed), _p(res["accept_len"]), _p(res["out_tokens"]),
                          _p(res["n_out"]), _p(res["band"]), _p(res["gap"]), _p(res["fallback"]),
                          nthreads or default_threads())
    _check(rc, "verify")
    return res


# ------------------------------------------------------------------------------ variants

def draft_greedy(U, W1, W2, anchor, nthreads: Optional[int] = None):
    """Greedy draft: x_k = argmax z (ties to the smallest v), q_tok = 1.

    Returns dict(tokens, q_tok, row_max, row_sumexp, gap) with [n, gamma] arrays (gap is
    the top-two logit gap)."""
    U = _c(U, np.float32)
    n, gamma, V = U.shape
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    r = W1.shape[1]
    assert W1.shape == (V, r) and W2.shape == (r, V)
    anchor = _c(anchor, np.int32)
    out = {k: np.zeros((n, gamma), dtype=np.float64) for k in ("q_tok", "row_max", "row_sumexp", "gap")}
    tokens = np.zeros((n, gamma), dtype=np.int32)
    rc = lib().dso_draft_greedy(_p(U), _p(W1), _p(W2), _p(anchor), n, gamma, V, r, _p(tokens),
                                _p(out["q_tok"]), _p(out["row_max"]), _p(out["row_sumexp"]),
                                _p(out["gap"]), nthreads or default_threads())
    _check(rc, "draft_greedy")
    out["tokens"] = tokens
    return out


def verify_greedy(T, tokens, ell, seed: int, req_ids: Optional[Sequence[int]] = None,
                  nthreads: Optional[int] = None):
    """Verification of greedily drafted tokens (proposal = point mass at each token).

    Same outputs as ``verify``."""
    T = _c(T, np.float32)
    n, g1, V = T.shape
    gamma = g1 - 1
    tokens = _c(tokens, np.int32)
    assert tokens.shape == (n, gamma)
    ids = _c(np.arange(n) if req_ids is None else req_ids, np.int32)
    res = dict(accept_len=np.zeros(n, np.int32), out_tokens=np.zeros((n, gamma + 1), np.int32),
               n_out=np.zeros(n, np.int32), band=np.zeros((n, gamma), np.float64),
               gap=np.zeros(n, np.float64), fallback=np.zeros(n, np.int32))
    rc = lib().dso_verify_greedy(_p(T), _p(tokens), _p(_c(ell, np.int32)), _p(ids), n, gamma, V,
                                 ctypes.c_uint64(seed), _p(res["accept_len"]),
                                 _p(res["out_tokens"]), _p(res["n_out"]), _p(res["band"]),
                                 _p(res["gap"]), _p(res["fallback"]), nthreads or default_threads())
    _check(rc, "verify_greedy")
    return res


def schedule_async(a, sps, K_in: int):
    """Two-step capacity scheduler: the first K_in items of this step's order (K_in < 0:
    this step's own early-stop count).  Returns (ell [R], B_total, Theta, K_out)."""
    a = _c(a, np.float32)
    R, gamma = a.shape
    sps = _c(sps, np.float32)
    ell = np.zeros(R, dtype=np.int32)
    Bt = np.zeros(1, dtype=np.int32)
    th = np.zeros(1, dtype=np.float64)
    ko = np.zeros(1, dtype=np.int32)
    rc = lib().dso_schedule_async(_p(a), R, gamma, _p(sps), len(sps), int(K_in), _p(ell), _p(Bt),
                                  _p(th), _p(ko))
    _check(rc, "schedule_async")
    return ell, int(Bt[0]), float(th[0]), int(ko[0])


def schedule_threshold(a, threshold: float):
    """Fixed-threshold truncation: l_r = leading run of a[r, j] > threshold.

    Returns (ell [R], B_total)."""
    a = _c(a, np.float32)
    R, gamma = a.shape
    ell = np.zeros(R, dtype=np.int32)
    Bt = np.zeros(1, dtype=np.int32)
    rc = lib().dso_schedule_threshold(_p(a), R, gamma, ctypes.c_float(threshold), _p(ell), _p(Bt))
    _check(rc, "schedule_threshold")
    return ell, int(Bt[0])


# ------------------------------------------------------------------------------ RNN head

def rnn_project(h, W_rnn, b_rnn):
    """hp [n, 3r] = h [n, H] W_rnn[2r:] + b_rnn in fp64 (h may be [B, gamma, H])."""
    h = _c(h, np.float32)
    lead = h.shape[:-1]
    H = h.shape[-1]
    W_rnn = _c(W_rnn, np.uint16)
    r = W_rnn.shape[1] // 3
    assert W_rnn.shape == (2 * r + H, 3 * r)
    n = int(np.prod(lead))
    hp = np.zeros((n, 3 * r), dtype=np.float64)
    _check(lib().dso_rnn_project(_p(h), _p(W_rnn), _p(_c(b_rnn, np.float32)), n, H, r, _p(hp)),
           "rnn_project")
    return hp.reshape(lead + (3 * r,))


def draft_rnn(U, h, W1, W2, W_rnn, b_rnn, anchor, seed: int, greedy: bool = False,
              req_ids: Optional[Sequence[int]] = None, nthreads: Optional[int] = None):
    """Draft with the RNN head.  Returns dict(tokens, q_tok, row_max, row_sumexp, gap,
    E [n, gamma, r] (tanh(output) rows), state [n, r])."""
    U = _c(U, np.float32)
    n, gamma, V = U.shape
    h = _c(h, np.float32)
    H = h.shape[2]
    W1 = _c(W1, np.uint16)
    W2 = _c(W2, np.uint16)
    r = W1.shape[1]
    W_rnn = _c(W_rnn, np.uint16)
    assert W_rnn.shape == (2 * r + H, 3 * r) and h.shape == (n, gamma, H)
    ids = _c(np.arange(n) if req_ids is None else req_ids, np.int32)
    out = {k: np.zeros((n, gamma), dtype=np.float64) for k in ("q_tok", "row_max", "row_sumexp", "gap")}
    tokens = np.zeros((n, gamma), dtype=np.int32)
    E = np.zeros((n, gamma, r), dtype=np.float64)
    state = np.zeros((n, r), dtype=np.float64)
    rc = lib().dso_draft_rnn(_p(U), _p(h), _p(W1), _p(W2), _p(W_rnn), _p(_c(b_rnn, np.float32)),
                             _p(_c(anchor, np.int32)), _p(ids), n, gamma, V, r, H,
                             ctypes.c_uint64(seed), int(bool(greedy)), _p(tokens), _p(out["q_tok"]),
                             _p(out["row_max"]), _p(out["row_sumexp"]), _p(out["gap"]), _p(E),
                             _p(state), nthreads or default_threads())
    _check(rc, "draft_rnn")
    out.update(tokens=tokens, E=E, state=state)
    return out


def verify_rnn(T, U, E, W2, tokens, ell, seed: int, req_ids: Optional[Sequence[int]] = None,
               nthreads: Optional[int] = None):
    """Verification of an RNN-head draft (proposal softmax(U + E W2)); outputs as verify."""
    T = _c(T, np.float32)
    U = _c(U, np.float32)
    n, gamma, V = U.shape
    E = _c(E, np.float64)
    r = E.shape[2]
    W2 = _c(W2, np.uint16)
    ids = _c(np.arange(n) if req_ids is None else req_ids, np.int32)
    res = dict(accept_len=np.zeros(n, np.int32), out_tokens=np.zeros((n, gamma + 1), np.int32),
               n_out=np.zeros(n, np.int32), band=np.zeros((n, gamma), np.float64),
               gap=np.zeros(n, np.float64), fallback=np.zeros(n, np.int32))
    rc = lib().dso_verify_rnn(_p(T), _p(U), _p(E), _p(W2), _p(_c(tokens, np.int32)),
                              _p(_c(ell, np.int32)), _p(ids), n, gamma, V, r, ctypes.c_uint64(seed),
                              _p(res["accept_len"]), _p(res["out_tokens"]), _p(res["n_out"]),
                              _p(res["band"]), _p(res["gap"]), _p(res["fallback"]),
                              nthreads or default_threads())
    _check(rc, "verify_rnn")
    return res


def step(inp, seed: int, nthreads: Optional[int] = None):
    """One full step (draft -> confidence -> schedule -> verify) on workload inputs.

    ``inp`` must hold every request (the scheduler is global)."""
    d = draft(inp.U, inp.W1, inp.W2, inp.anchor, seed, inp.requests, nthreads)
    c, a = confidence(inp.h, inp.anchor, d["tokens"], inp.W1, inp.w_c, float(inp.b_c))
    ell, Bt, th = schedule(a.astype(np.float32), inp.sps)
    v = verify(inp.T, inp.U, inp.W1, inp.W2, inp.anchor, d["tokens"], ell, seed, inp.requests, nthreads)
    return dict(draft=d, c=c, a=a, ell=ell, B_total=Bt, theta=th, verify=v)
