"""DSpark per-step hot path on one GB300 (sm_103a): Python binding of libdspark.

The library behind this binding (``include/dspark.h``) holds the four calls of one
speculative step -- ``dspark_draft``, ``dspark_confidence``, ``dspark_schedule``,
``dspark_verify`` -- plus ``dspark_draft_confidence_schedule`` (the first three in one
launch), ``dspark_markov_bias``, the packed-W2 variants of the draft and the verification,
greedy drafting with its verification, the asynchronous two-step capacity scheduler,
fixed-threshold truncation and the RNN head; every step of the computation runs in its
CUDA kernels.  This module only marshals arguments: it passes device pointers of
torch tensors and the current CUDA stream through ctypes, and allocates outputs and the
workspace with torch.  There is no CPU fallback: without the built library and a CUDA
device every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

from . import _build

STATUS = {0: "DSPARK_OK", 1: "DSPARK_ERR_INVALID_ARG", 2: "DSPARK_ERR_UNSUPPORTED",
          3: "DSPARK_ERR_CUDA", 4: "DSPARK_ERR_TIMEOUT", 5: "DSPARK_ERR_DEVICE_CHECK"}

# (name, restype, argtypes) of every exported symbol, in header order
_P, _I, _U64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = [
    ("dspark_status_string", ctypes.c_char_p, [_I]),
    ("dspark_workspace_bytes", _SZ, [_I, _I, _I, _I, _I]),
    ("dspark_markov_bias", _I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    ("dspark_packed_w2_bytes", _SZ, [_I, _I]),
    ("dspark_pack_w2", _I, [_P, _I, _I, _P, _SZ, _P]),
    ("dspark_draft_packed", _I, [_P, _P, _P, _P, _I, _I, _I, _I, _U64, _P, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_draft", _I, [_P, _P, _P, _P, _I, _I, _I, _I, _U64, _P, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_confidence", _I, [_P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    ("dspark_confidence_schedule", _I, [_P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _P, _I, _P, _P,
                                        _P, _P, _P, _P, _SZ, _P]),
    ("dspark_schedule", _I, [_P, _I, _I, _P, _I, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_verify", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _U64,
                           _P, _P, _P, _P, _SZ, _P]),
    ("dspark_verify_packed", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _U64,
                                  _P, _P, _P, _P, _SZ, _P]),
    ("dspark_draft_noalloc", _I, [_P, _P, _P, _P, _I, _I, _I, _I, _U64, _P, _P, _P, _P, _P]),
    ("dspark_draft_greedy", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_verify_greedy", _I, [_P, _P, _P, _I, _I, _I, _U64, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_schedule_async", _I, [_P, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_schedule_threshold", _I, [_P, _I, _I, _F, _P, _P, _P]),
    ("dspark_rnn_packed_bytes", _SZ, [_I]),
    ("dspark_rnn_pack", _I, [_P, _I, _P, _SZ, _P]),
    ("dspark_rnn_project", _I, [_P, _P, _P, _I, _I, _I, _I, _P, _P]),
    ("dspark_draft_rnn", _I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _U64, _I, _P, _P, _P, _P,
                              _P, _P, _SZ, _P]),
    ("dspark_verify_rnn", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _U64, _P, _P,
                               _P, _P, _SZ, _P]),
    ("dspark_last_device_status", _I, [_P, _P]),
    ("dspark_draft_confidence_schedule", _I, [_P, _P, _P, _P, _P, _P, _F, _P, _I, _I, _I, _I, _I, _I,
                                              _U64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    ("dspark_testing_set_wait_limit", None, [ctypes.c_longlong, _I]),
    ("dspark_copy_target_rows", _I, [_P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
]

_lib = None


class DSparkError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call} failed: {STATUS.get(code, code)}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libdspark.so (building it in-tree first when it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build() if build_if_missing else _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"libdspark.so is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("the DSpark kernels need a CUDA device; there is no CPU fallback")
    return torch


def _ptr(t) -> int:
    return t.data_ptr()


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(call: str, code: int):
    if code != 0:
        raise DSparkError(call, code)


def workspace_bytes(B: int, gamma: int, V: int, r: int, H: int = 0) -> int:
    n = lib().dspark_workspace_bytes(B, gamma, V, r, H)
    if n == 0:
        raise ValueError(f"unsupported shapes B={B} gamma={gamma} V={V} r={r} H={H}")
    return int(n)


class Workspace:
    """Caller-owned scratch for the calls (zero-filled, 256-byte aligned torch buffer)."""

    def __init__(self, B: int, gamma: int, V: int, r: int, H: int = 0, device="cuda"):
        torch = _torch()
        self.nbytes = workspace_bytes(B, gamma, V, r, H)
        self.buf = torch.zeros(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off

    def status(self, stream=None) -> int:
        return int(lib().dspark_last_device_status(ctypes.c_void_p(self.ptr), _stream(stream)))


def as_bf16_tensor(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 tensor on ``device``."""
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def testing_set_wait_limit(wait_cycles: int = 0, unreachable_barrier: bool = False):
    """Bound of the draft kernels' waits (SM cycles, 0: the default of about 2 s) and, when
    ``unreachable_barrier``, barriers that cannot complete, for the draft launches that
    follow (tests of the timeout path; ``testing_set_wait_limit()`` restores the production
    setting)."""
    lib().dspark_testing_set_wait_limit(int(wait_cycles), int(bool(unreachable_barrier)))


# ------------------------------------------------------------------------------ calls

def markov_bias(W1, W2, prev, ws: Workspace, out=None, prev_stride: int = 1, stream=None):
    torch = _torch()
    V, r = W1.shape
    B = (prev.numel() + prev_stride - 1) // prev_stride
    if out is None:
        out = torch.empty((B, V), dtype=torch.float32, device=W1.device)
    _check("dspark_markov_bias", lib().dspark_markov_bias(
        _ptr(W1), _ptr(W2), _ptr(prev), prev_stride, B, V, r, _ptr(out),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def draft(U, W1, W2, anchor, seed: int, ws: Workspace, out: Optional[Dict] = None, stream=None):
    torch = _torch()
    B, gamma, V = U.shape
    r = W1.shape[1]
    if out is None:
        out = dict(tokens=torch.empty((B, gamma), dtype=torch.int32, device=U.device),
                   q_tok=torch.empty((B, gamma), dtype=torch.float32, device=U.device),
                   row_max=torch.empty((B, gamma), dtype=torch.float32, device=U.device),
                   row_sumexp=torch.empty((B, gamma), dtype=torch.float32, device=U.device))
    _check("dspark_draft", lib().dspark_draft(
        _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchor), B, gamma, V, r, ctypes.c_uint64(seed),
        _ptr(out["tokens"]), _ptr(out["q_tok"]), _ptr(out["row_max"]), _ptr(out["row_sumexp"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def pack_w2(W2, stream=None):
    """Packed copy of W2 [r, V] for draft_packed (a device tensor; done once per weights)."""
    torch = _torch()
    r, V = W2.shape
    n = lib().dspark_packed_w2_bytes(V, r)
    if n == 0:
        raise ValueError(f"unsupported shapes V={V} r={r}")
    W2p = torch.empty(n // 2, dtype=torch.bfloat16, device=W2.device)
    _check("dspark_pack_w2", lib().dspark_pack_w2(_ptr(W2), V, r, _ptr(W2p), n, _stream(stream)))
    return W2p


def draft_packed(U, W1, W2p, anchor, seed: int, ws: Workspace, out: Optional[Dict] = None,
                 stream=None):
    torch = _torch()
    B, gamma, V = U.shape
    r = W1.shape[1]
    if out is None:
        out = dict(tokens=torch.empty((B, gamma), dtype=torch.int32, device=U.device),
                   q_tok=torch.empty((B, gamma), dtype=torch.float32, device=U.device),
                   row_max=torch.empty((B, gamma), dtype=torch.float32, device=U.device),
                   row_sumexp=torch.empty((B, gamma), dtype=torch.float32, device=U.device))
    _check("dspark_draft_packed", lib().dspark_draft_packed(
        _ptr(U), _ptr(W1), _ptr(W2p), _ptr(anchor), B, gamma, V, r, ctypes.c_uint64(seed),
        _ptr(out["tokens"]), _ptr(out["q_tok"]), _ptr(out["row_max"]), _ptr(out["row_sumexp"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def confidence(h, anchor, tokens, W1, w_c, b_c: float, ws: Workspace, out=None, stream=None):
    torch = _torch()
    B, gamma, H = h.shape
    V, r = W1.shape
    if out is None:
        out = (torch.empty((B, gamma), dtype=torch.float32, device=h.device),
               torch.empty((B, gamma), dtype=torch.float32, device=h.device))
    c, a = out
    _check("dspark_confidence", lib().dspark_confidence(
        _ptr(h), _ptr(anchor), _ptr(tokens), _ptr(W1), _ptr(w_c), ctypes.c_float(b_c), B, gamma,
        H, r, V, _ptr(c), _ptr(a), ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return c, a


def confidence_schedule(h, anchor, tokens, W1, w_c, b_c: float, sps, ws: Workspace, conf_out=None,
                        sched_out=None, stream=None):
    """confidence and schedule in one launch (the last CTA schedules)."""
    torch = _torch()
    B, gamma, H = h.shape
    V, r = W1.shape
    if conf_out is None:
        conf_out = (torch.empty((B, gamma), dtype=torch.float32, device=h.device),
                    torch.empty((B, gamma), dtype=torch.float32, device=h.device))
    if sched_out is None:
        sched_out = (torch.empty(B, dtype=torch.int32, device=h.device),
                     torch.empty(1, dtype=torch.int32, device=h.device),
                     torch.empty(1, dtype=torch.float64, device=h.device))
    c, a = conf_out
    ell, Bt, th = sched_out
    _check("dspark_confidence_schedule", lib().dspark_confidence_schedule(
        _ptr(h), _ptr(anchor), _ptr(tokens), _ptr(W1), _ptr(w_c), ctypes.c_float(b_c), B, gamma,
        H, r, V, _ptr(sps), sps.numel(), _ptr(c), _ptr(a), _ptr(ell), _ptr(Bt), _ptr(th),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return (c, a), (ell, Bt, th)


def draft_confidence_schedule(U, W1, W2p, anchor, h, w_c, b_c: float, sps, seed: int, ws: Workspace,
                              draft_out: Optional[Dict] = None, conf_out=None, sched_out=None,
                              stream=None):
    """draft (packed W2), confidence, survival and schedule in one launch (two when
    B * gamma > 4096: the scheduler kernel follows)."""
    torch = _torch()
    B, gamma, V = U.shape
    r = W1.shape[1]
    H = h.shape[2]
    if draft_out is None:
        draft_out = _draft_outputs(B, gamma, U.device)
    if conf_out is None:
        conf_out = (torch.empty((B, gamma), dtype=torch.float32, device=U.device),
                    torch.empty((B, gamma), dtype=torch.float32, device=U.device))
    if sched_out is None:
        sched_out = (torch.empty(B, dtype=torch.int32, device=U.device),
                     torch.empty(1, dtype=torch.int32, device=U.device),
                     torch.empty(1, dtype=torch.float64, device=U.device))
    c, a = conf_out
    ell, Bt, th = sched_out
    _check("dspark_draft_confidence_schedule", lib().dspark_draft_confidence_schedule(
        _ptr(U), _ptr(W1), _ptr(W2p), _ptr(anchor), _ptr(h), _ptr(w_c), ctypes.c_float(b_c),
        _ptr(sps), sps.numel(), B, gamma, V, r, H, ctypes.c_uint64(seed),
        _ptr(draft_out["tokens"]), _ptr(draft_out["q_tok"]), _ptr(draft_out["row_max"]),
        _ptr(draft_out["row_sumexp"]), _ptr(c), _ptr(a), _ptr(ell), _ptr(Bt), _ptr(th),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return draft_out, (c, a), (ell, Bt, th)


def copy_target_rows(T_src, T, ell, ws: Workspace, stream=None):
    """T[b, j] for j <= ell[b] (the rows a verification under schedule ell reads) from
    T_src into the device tensor T ([B, gamma + 1, V] fp32 both).  T_src may be a pinned
    host tensor: a kernel reads the rows over the host link."""
    B, g1, V = T.shape
    _check("dspark_copy_target_rows", lib().dspark_copy_target_rows(
        _ptr(T_src), _ptr(T), _ptr(ell), B, g1 - 1, V, ctypes.c_void_p(ws.ptr), ws.nbytes,
        _stream(stream)))
    return T


def schedule(a, sps, ws: Workspace, out=None, stream=None):
    torch = _torch()
    R, gamma = a.shape
    if out is None:
        out = (torch.empty(R, dtype=torch.int32, device=a.device),
               torch.empty(1, dtype=torch.int32, device=a.device),
               torch.empty(1, dtype=torch.float64, device=a.device))
    ell, Bt, th = out
    _check("dspark_schedule", lib().dspark_schedule(
        _ptr(a), R, gamma, _ptr(sps), sps.numel(), _ptr(ell), _ptr(Bt), _ptr(th),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return ell, Bt, th


def verify(T, U, W1, W2, anchor, tokens, q_tok, row_max, row_sumexp, ell, seed: int,
           ws: Workspace, out: Optional[Dict] = None, stream=None):
    torch = _torch()
    B, gamma, V = U.shape
    r = W1.shape[1]
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=U.device),
                   out_tokens=torch.empty((B, gamma + 1), dtype=torch.int32, device=U.device),
                   n_out=torch.empty(B, dtype=torch.int32, device=U.device))
    _check("dspark_verify", lib().dspark_verify(
        _ptr(T), _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchor), _ptr(tokens), _ptr(q_tok),
        _ptr(row_max), _ptr(row_sumexp), _ptr(ell), B, gamma, V, r, ctypes.c_uint64(seed),
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["n_out"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def verify_packed(T, U, W1, W2p, anchor, tokens, q_tok, row_max, row_sumexp, ell, seed: int,
                  ws: Workspace, out: Optional[Dict] = None, stream=None):
    """verify with the packed W2 of pack_w2 (the copy draft_packed streams)."""
    torch = _torch()
    B, gamma, V = U.shape
    r = W1.shape[1]
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=U.device),
                   out_tokens=torch.empty((B, gamma + 1), dtype=torch.int32, device=U.device),
                   n_out=torch.empty(B, dtype=torch.int32, device=U.device))
    _check("dspark_verify_packed", lib().dspark_verify_packed(
        _ptr(T), _ptr(U), _ptr(W1), _ptr(W2p), _ptr(anchor), _ptr(tokens), _ptr(q_tok),
        _ptr(row_max), _ptr(row_sumexp), _ptr(ell), B, gamma, V, r, ctypes.c_uint64(seed),
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["n_out"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def _draft_outputs(B, gamma, device):
    torch = _torch()
    return dict(tokens=torch.empty((B, gamma), dtype=torch.int32, device=device),
                q_tok=torch.empty((B, gamma), dtype=torch.float32, device=device),
                row_max=torch.empty((B, gamma), dtype=torch.float32, device=device),
                row_sumexp=torch.empty((B, gamma), dtype=torch.float32, device=device))


def _verify_outputs(B, gamma, device):
    torch = _torch()
    return dict(accept_len=torch.empty(B, dtype=torch.int32, device=device),
                out_tokens=torch.empty((B, gamma + 1), dtype=torch.int32, device=device),
                n_out=torch.empty(B, dtype=torch.int32, device=device))


def draft_greedy(U, W1, W2, anchor, ws: Workspace, out: Optional[Dict] = None, packed: bool = False,
                 stream=None):
    """Greedy draft (x_k = argmax z_k, q_tok = 1).  ``W2`` is the [r, V] matrix, or the
    packed copy of pack_w2 when ``packed``."""
    B, gamma, V = U.shape
    r = W1.shape[1]
    if out is None:
        out = _draft_outputs(B, gamma, U.device)
    w2, w2p = (None, W2) if packed else (W2, None)
    _check("dspark_draft_greedy", lib().dspark_draft_greedy(
        _ptr(U), _ptr(W1), None if w2 is None else _ptr(w2), None if w2p is None else _ptr(w2p),
        _ptr(anchor), B, gamma, V, r,
        _ptr(out["tokens"]), _ptr(out["q_tok"]), _ptr(out["row_max"]), _ptr(out["row_sumexp"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def verify_greedy(T, tokens, ell, seed: int, ws: Workspace, out: Optional[Dict] = None,
                  stream=None):
    """Verification of greedily drafted tokens (point-mass proposals)."""
    B, g1, V = T.shape
    gamma = g1 - 1
    if out is None:
        out = _verify_outputs(B, gamma, T.device)
    _check("dspark_verify_greedy", lib().dspark_verify_greedy(
        _ptr(T), _ptr(tokens), _ptr(ell), B, gamma, V, ctypes.c_uint64(seed),
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["n_out"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def schedule_async(a, sps, K_in, K_out, ws: Workspace, out=None, stream=None):
    """Two-step capacity scheduler: admits the first ``*K_in`` items of this step's order
    (``K_in`` None or holding a negative value: this step's own early-stop count) and
    writes that count to ``K_out`` (device int32 tensors of one element; may be the same
    tensor, or None)."""
    torch = _torch()
    R, gamma = a.shape
    if out is None:
        out = (torch.empty(R, dtype=torch.int32, device=a.device),
               torch.empty(1, dtype=torch.int32, device=a.device),
               torch.empty(1, dtype=torch.float64, device=a.device))
    ell, Bt, th = out
    _check("dspark_schedule_async", lib().dspark_schedule_async(
        _ptr(a), R, gamma, _ptr(sps), sps.numel(), None if K_in is None else _ptr(K_in),
        None if K_out is None else _ptr(K_out), _ptr(ell), _ptr(Bt), _ptr(th),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return ell, Bt, th


class CapacityRing:
    """The two device words of the two-step pipeline: step t reads slot t % 2 (written at
    step t - 2) and overwrites it with its own early-stop count.  Both start at -1, so
    the first two steps admit their own count."""

    def __init__(self, device="cuda"):
        torch = _torch()
        self.slots = torch.full((2,), -1, dtype=torch.int32, device=device)

    def slot(self, t: int):
        return self.slots[t % 2:t % 2 + 1]


def schedule_threshold(a, threshold: float, out=None, stream=None):
    """Fixed-threshold truncation: ell[r] = leading positions with a[r, j] > threshold."""
    torch = _torch()
    R, gamma = a.shape
    if out is None:
        out = (torch.empty(R, dtype=torch.int32, device=a.device),
               torch.empty(1, dtype=torch.int32, device=a.device))
    ell, Bt = out
    _check("dspark_schedule_threshold", lib().dspark_schedule_threshold(
        _ptr(a), R, gamma, ctypes.c_float(threshold), _ptr(ell), _ptr(Bt), _stream(stream)))
    return ell, Bt


def rnn_pack(W_rnn, r: int, stream=None):
    """Transposed recurrent rows of the RNN head's layer (once per weights)."""
    torch = _torch()
    n = lib().dspark_rnn_packed_bytes(r)
    if n == 0:
        raise ValueError(f"unsupported rank r={r}")
    Wrec = torch.empty(n // 2, dtype=torch.bfloat16, device=W_rnn.device)
    _check("dspark_rnn_pack", lib().dspark_rnn_pack(_ptr(W_rnn), r, _ptr(Wrec), n, _stream(stream)))
    return Wrec


def rnn_project(h, W_rnn, b_rnn, out=None, stream=None):
    """hp [B, gamma, 3r] = h W_rnn[2r:] + b_rnn (the token-independent part of the layer)."""
    torch = _torch()
    B, gamma, H = h.shape
    r = W_rnn.shape[1] // 3
    if out is None:
        out = torch.empty((B, gamma, 3 * r), dtype=torch.float32, device=h.device)
    _check("dspark_rnn_project", lib().dspark_rnn_project(
        _ptr(h), _ptr(W_rnn), _ptr(b_rnn), B, gamma, H, r, _ptr(out), _stream(stream)))
    return out


def draft_rnn(U, W1, W2, Wrec, hp, anchor, seed: int, ws: Workspace, greedy: bool = False,
              packed: bool = False, out: Optional[Dict] = None, stream=None):
    """Draft with the RNN head; ``out`` also gets ``E`` [B, gamma, r] (tanh(output) rows)."""
    torch = _torch()
    B, gamma, V = U.shape
    r = W1.shape[1]
    if out is None:
        out = _draft_outputs(B, gamma, U.device)
    if "E" not in out:
        out["E"] = torch.empty((B, gamma, r), dtype=torch.float32, device=U.device)
    w2, w2p = (None, W2) if packed else (W2, None)
    _check("dspark_draft_rnn", lib().dspark_draft_rnn(
        _ptr(U), _ptr(W1), None if w2 is None else _ptr(w2), None if w2p is None else _ptr(w2p),
        _ptr(Wrec), _ptr(hp), _ptr(anchor), B, gamma, V, r, ctypes.c_uint64(seed), int(bool(greedy)),
        _ptr(out["tokens"]), _ptr(out["q_tok"]), _ptr(out["row_max"]), _ptr(out["row_sumexp"]),
        _ptr(out["E"]), ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


def verify_rnn(T, U, E, W2, tokens, q_tok, row_max, row_sumexp, ell, seed: int, ws: Workspace,
               packed: bool = False, out: Optional[Dict] = None, stream=None):
    """Verification of a Gumbel-sampled RNN draft (``E`` from draft_rnn)."""
    B, gamma, V = U.shape
    r = E.shape[2]
    if out is None:
        out = _verify_outputs(B, gamma, U.device)
    w2, w2p = (None, W2) if packed else (W2, None)
    _check("dspark_verify_rnn", lib().dspark_verify_rnn(
        _ptr(T), _ptr(U), _ptr(E), None if w2 is None else _ptr(w2), None if w2p is None else _ptr(w2p),
        _ptr(tokens), _ptr(q_tok), _ptr(row_max), _ptr(row_sumexp), _ptr(ell), B, gamma, V, r,
        ctypes.c_uint64(seed), _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["n_out"]),
        ctypes.c_void_p(ws.ptr), ws.nbytes, _stream(stream)))
    return out


# ------------------------------------------------------------------------ whole step

class Step:
    """One speculative step (draft -> confidence -> schedule -> verify) with preallocated
    outputs and workspace, so that ``run`` launches kernels only (capturable in a CUDA
    graph).  ``dev`` maps input names (U, T, W1, W2, h, w_c, anchor, sps) to device
    tensors; ``b_c`` is the confidence-head bias.

    ``sampling``: "gumbel" (the draft samples from q_k) or "greedy" (argmax drafts, verified
    as point-mass proposals).  ``head``: "markov" or "rnn" (``dev`` then also holds W_rnn
    and b_rnn; each step first projects the hidden states).  ``scheduler``: "theta" (the early-stop scheduler), "async"
    (the two-step capacity scheduler; ``run(seed, t=...)`` picks the ring slot of step t)
    or "threshold" (fixed truncation at ``threshold``).  ``fused``: the default step
    (Gumbel, Markov head, early-stop scheduler, packed W2) drafts, scores confidence and
    schedules in one launch (``draft_confidence_schedule``); False runs the calls one by one."""

    SAMPLING = ("gumbel", "greedy")
    HEADS = ("markov", "rnn")
    SCHEDULERS = ("theta", "async", "threshold")

    def __init__(self, dev: Dict, b_c: float, ws: Optional[Workspace] = None, packed: bool = True,
                 sampling: str = "gumbel", scheduler: str = "theta", threshold: float = 0.5,
                 W2p=None, head: str = "markov", fused: bool = True):
        torch = _torch()
        if sampling not in self.SAMPLING or scheduler not in self.SCHEDULERS or head not in self.HEADS:
            raise ValueError(f"sampling {sampling!r} / scheduler {scheduler!r} / head {head!r}")
        self.head = head
        self.sampling, self.scheduler, self.threshold = sampling, scheduler, float(threshold)
        self.dev = dev
        # the draft streams W2 from a packed copy made once here (weight preparation), or
        # from the copy ``W2p`` of an earlier pack_w2 call
        self.W2p = (W2p if W2p is not None else pack_w2(dev["W2"])) if packed else None
        self.b_c = float(b_c)
        B, gamma, V = dev["U"].shape
        r = dev["W1"].shape[1]
        H = dev["h"].shape[2]
        self.shape = (B, gamma, V, r, H)
        self.ws = ws or Workspace(B, gamma, V, r, H, device=dev["U"].device)
        d = dev["U"].device
        f32, i32 = torch.float32, torch.int32
        self.draft_out = dict(tokens=torch.empty((B, gamma), dtype=i32, device=d),
                              q_tok=torch.empty((B, gamma), dtype=f32, device=d),
                              row_max=torch.empty((B, gamma), dtype=f32, device=d),
                              row_sumexp=torch.empty((B, gamma), dtype=f32, device=d))
        self.conf_out = (torch.empty((B, gamma), dtype=f32, device=d),
                         torch.empty((B, gamma), dtype=f32, device=d))
        self.sched_out = (torch.empty(B, dtype=i32, device=d), torch.empty(1, dtype=i32, device=d),
                          torch.empty(1, dtype=torch.float64, device=d))
        self.verify_out = dict(accept_len=torch.empty(B, dtype=i32, device=d),
                               out_tokens=torch.empty((B, gamma + 1), dtype=i32, device=d),
                               n_out=torch.empty(B, dtype=i32, device=d))
        self.ring = CapacityRing(d) if scheduler == "async" else None
        # the default step (Gumbel drafts, the Markov head, the early-stop scheduler, packed
        # W2) drafts, scores confidence and schedules in one launch
        # (the draft grid keeps the survivals of 512 requests per CTA and holds at least
        # min(vocabulary tiles, 148) CTAs on a GB300)
        self.fused = (fused and sampling == "gumbel" and head == "markov" and scheduler == "theta"
                      and self.W2p is not None and B * gamma <= 16384
                      and B <= 512 * min((V + 127) // 128, 148))
        if head == "rnn":
            self.Wrec = rnn_pack(dev["W_rnn"], r)
            self.hp = torch.empty((B, gamma, 3 * r), dtype=f32, device=d)
            self.draft_out["E"] = torch.empty((B, gamma, r), dtype=f32, device=d)

    def run(self, seed: int, stream=None, t: int = 0, T_host=None):
        """One step.  T_host: the step's target logits in host memory (pinned); then only
        the rows the verification reads (T[b, j], j <= l_b) are fetched into dev["T"], once
        the schedule is known."""
        x = self.dev
        B, gamma = x["U"].shape[:2]
        if self.fused:
            # draft, confidence, survival and schedule in one launch, then verification
            d, (ell, _, _) = self.first_launch(seed, stream)
            if T_host is not None:
                copy_target_rows(T_host, x["T"], ell, self.ws, stream)
            verify_packed(x["T"], x["U"], x["W1"], self.W2p, x["anchor"], d["tokens"], d["q_tok"],
                          d["row_max"], d["row_sumexp"], ell, seed, self.ws, self.verify_out, stream)
            return self
        d = self.draft(seed, stream)
        if self.scheduler == "theta" and B * gamma <= 16384:
            # the early-stop scheduler runs in the confidence kernel's last CTA
            _, (ell, _, _) = confidence_schedule(x["h"], x["anchor"], d["tokens"], x["W1"], x["w_c"],
                                                 self.b_c, x["sps"], self.ws, self.conf_out,
                                                 self.sched_out, stream)
        else:
            c, a = confidence(x["h"], x["anchor"], d["tokens"], x["W1"], x["w_c"], self.b_c, self.ws,
                              self.conf_out, stream)
            ell = self._schedule(a, stream, t)
        if T_host is not None:
            copy_target_rows(T_host, x["T"], ell, self.ws, stream)
        if self.sampling == "greedy":
            verify_greedy(x["T"], d["tokens"], ell, seed, self.ws, self.verify_out, stream)
        elif self.head == "rnn":
            packed = self.W2p is not None
            verify_rnn(x["T"], x["U"], d["E"], self.W2p if packed else x["W2"], d["tokens"],
                       d["q_tok"], d["row_max"], d["row_sumexp"], ell, seed, self.ws, packed,
                       self.verify_out, stream)
        elif self.W2p is not None:
            verify_packed(x["T"], x["U"], x["W1"], self.W2p, x["anchor"], d["tokens"], d["q_tok"],
                          d["row_max"], d["row_sumexp"], ell, seed, self.ws, self.verify_out, stream)
        else:
            verify(x["T"], x["U"], x["W1"], x["W2"], x["anchor"], d["tokens"], d["q_tok"],
                   d["row_max"], d["row_sumexp"], ell, seed, self.ws, self.verify_out, stream)
        return self

    def first_launch(self, seed: int, stream=None):
        """The fused step's first launch alone: draft, confidence and schedule."""
        x = self.dev
        d, _, sched = draft_confidence_schedule(
            x["U"], x["W1"], self.W2p, x["anchor"], x["h"], x["w_c"], self.b_c, x["sps"], seed,
            self.ws, self.draft_out, self.conf_out, self.sched_out, stream)
        return d, sched

    def draft(self, seed: int, stream=None):
        """The draft call of the step alone (into the step's draft outputs)."""
        x = self.dev
        if self.head == "rnn":
            rnn_project(x["h"], x["W_rnn"], x["b_rnn"], self.hp, stream)
            packed = self.W2p is not None
            return draft_rnn(x["U"], x["W1"], self.W2p if packed else x["W2"], self.Wrec, self.hp,
                             x["anchor"], seed, self.ws, self.sampling == "greedy", packed,
                             self.draft_out, stream)
        if self.sampling == "greedy":
            w2, packed = (self.W2p, True) if self.W2p is not None else (x["W2"], False)
            return draft_greedy(x["U"], x["W1"], w2, x["anchor"], self.ws, self.draft_out, packed,
                                stream)
        if self.W2p is not None:
            return draft_packed(x["U"], x["W1"], self.W2p, x["anchor"], seed, self.ws,
                                self.draft_out, stream)
        return draft(x["U"], x["W1"], x["W2"], x["anchor"], seed, self.ws, self.draft_out, stream)

    def _schedule(self, a, stream, t: int):
        if self.scheduler == "async":
            k = self.ring.slot(t)
            ell, _, _ = schedule_async(a, self.dev["sps"], k, k, self.ws, self.sched_out, stream)
        elif self.scheduler == "threshold":
            ell, _ = schedule_threshold(a, self.threshold, self.sched_out[:2], stream)
        else:
            ell, _, _ = schedule(a, self.dev["sps"], self.ws, self.sched_out, stream)
        return ell

    def capture(self, seeds, draft_only: bool = False, first_only: bool = False):
        """CUDA graphs of run(seed) (or of the draft call alone, or of the fused step's
        first launch alone), one per seed.  The seed is a launch argument, so each graph
        replays with its own random stream.  With the two-step scheduler, graph i uses
        capacity slot i % 2."""
        torch = _torch()
        if first_only and not self.fused:
            raise ValueError("first_only needs the fused step")
        graphs = []
        for i, sd in enumerate(seeds):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                if first_only:
                    self.first_launch(sd)
                elif draft_only:
                    self.draft(sd)
                else:
                    self.run(sd, t=i)
            graphs.append(g)
        return graphs

    # per-step inputs (the backbone's and the target's outputs); the weights, the
    # confidence head and the SPS table stay resident on the device.  The target logits T
    # are fetched row by row by the step itself (only the rows it verifies); the others
    # are copied whole.
    STEP_INPUTS = ("U", "T", "h", "anchor")
    COPIED_INPUTS = ("U", "h", "anchor")
    STEP_OUTPUTS = ("out_tokens", "accept_len", "n_out")

    def pinned_host_buffers(self):
        """Pinned host tensors shaped like the per-step inputs and outputs."""
        torch = _torch()
        hin = {k: torch.empty(self.dev[k].shape, dtype=self.dev[k].dtype, pin_memory=True)
               for k in self.STEP_INPUTS}
        hout = {k: torch.empty(self.verify_out[k].shape, dtype=self.verify_out[k].dtype,
                               pin_memory=True) for k in self.STEP_OUTPUTS}
        return hin, hout

    def run_from_host(self, seed: int, host_in: Dict, host_out: Dict, stream=None):
        """One step from pinned host inputs to pinned host outputs: host->device copies of
        the step's inputs, the four calls, device->host copies of the verified tokens."""
        torch = _torch()
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            for k in self.COPIED_INPUTS:
                self.dev[k].copy_(host_in[k], non_blocking=True)
            self.run(seed, s, T_host=host_in["T"])
            for k in self.STEP_OUTPUTS:
                host_out[k].copy_(self.verify_out[k], non_blocking=True)
        return host_out

    def pipeline(self):
        """A HostPipeline over this step (see there)."""
        return HostPipeline(self)

    def step_bytes(self, B_total: Optional[float] = None):
        """(host->device, device->host) bytes of one run_from_host call: the copied inputs,
        plus the target rows fetched, B_total = sum_b (l_b + 1) rows of V fp32 (all
        B (gamma + 1) rows when B_total is None)."""
        h2d = sum(self.dev[k].numel() * self.dev[k].element_size() for k in self.COPIED_INPUTS)
        B, g1, V = self.dev["T"].shape
        h2d += (B * g1 if B_total is None else B_total) * V * self.dev["T"].element_size()
        d2h = sum(self.verify_out[k].numel() * self.verify_out[k].element_size() for k in self.STEP_OUTPUTS)
        return int(h2d), int(d2h)

    def results(self) -> Dict[str, np.ndarray]:
        out = {k: v.cpu().numpy() for k, v in self.draft_out.items()}
        if self.head == "rnn":
            out["hp"] = self.hp.cpu().numpy()
        out["c"], out["a"] = (t.cpu().numpy() for t in self.conf_out)
        out["ell"] = self.sched_out[0].cpu().numpy()
        out["B_total"] = int(self.sched_out[1].item())
        if self.scheduler != "threshold":
            out["theta"] = float(self.sched_out[2].item())
        out.update({k: v.cpu().numpy() for k, v in self.verify_out.items()})
        return out


class HostPipeline:
    """Steps fed from pinned host buffers, with the next step's host->device copies
    overlapped with the current step's kernels.

    The step's per-step inputs get a second device copy; step i reads input set i % 2,
    whose copies (U, h, anchor) run on a separate copy stream and are ordered before the
    step by an event, and step i + 2's copies into the same set wait for an event recorded
    after step i's kernels.  The target logits stay in host memory: step i fetches the
    rows it verifies into its set once its schedule is known (Step.run with T_host).  Every
    step's inputs still come from the host and every step's verified tokens are copied
    back, on the step's stream.  The step object is given its own dictionary of device
    tensors, so the caller's dictionary is unchanged.
    """

    def __init__(self, step: "Step"):
        torch = _torch()
        self.step = step
        step.dev = dict(step.dev)
        dev0 = {k: step.dev[k] for k in step.STEP_INPUTS}
        self.sets = [dev0, {k: torch.empty_like(v) for k, v in dev0.items()}]
        device = dev0["U"].device
        self.copy_stream = torch.cuda.Stream(device=device)
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.free = [torch.cuda.Event(), torch.cuda.Event()]

    def _copy_in(self, i: int, host_in: Dict):
        torch = _torch()
        b = i % 2
        with torch.cuda.stream(self.copy_stream):
            self.copy_stream.wait_event(self.free[b])
            for k in self.step.COPIED_INPUTS:
                self.sets[b][k].copy_(host_in[k], non_blocking=True)
            self.ready[b].record(self.copy_stream)

    def run(self, seeds, host_ins, host_outs, stream=None):
        """Steps i = 0.. with seed seeds[i], inputs host_ins[i] and outputs host_outs[i]
        (dicts of pinned tensors shaped like Step.pinned_host_buffers()); returns after
        enqueueing everything on `stream` (default: the current stream)."""
        torch = _torch()
        s = stream if stream is not None else torch.cuda.current_stream()
        n = len(seeds)
        if n == 0:
            return host_outs
        self._copy_in(0, host_ins[0])
        for i in range(n):
            if i + 1 < n:
                self._copy_in(i + 1, host_ins[i + 1])
            b = i % 2
            s.wait_event(self.ready[b])
            self.step.dev.update(self.sets[b])
            self.step.run(seeds[i], s, t=i, T_host=host_ins[i]["T"])
            self.free[b].record(s)
            with torch.cuda.stream(s):
                for k in self.step.STEP_OUTPUTS:
                    host_outs[i][k].copy_(self.step.verify_out[k], non_blocking=True)
        return host_outs


def to_device(inp, device="cuda") -> Dict:
    """Workload inputs (numpy, see the ``workloads`` module) -> device tensors."""
    torch = _torch()
    dev = dict(U=torch.from_numpy(inp.U).to(device), W1=as_bf16_tensor(inp.W1, device),
               W2=as_bf16_tensor(inp.W2, device), h=torch.from_numpy(inp.h).to(device),
               w_c=torch.from_numpy(inp.w_c).to(device),
               anchor=torch.from_numpy(inp.anchor).to(device),
               sps=torch.from_numpy(inp.sps).to(device))
    if inp.T is not None:
        dev["T"] = torch.from_numpy(inp.T).to(device)
    return dev


def rnn_to_device(W_rnn, b_rnn, dev: Dict, device="cuda") -> Dict:
    """Add the RNN head's weights (numpy bf16 bits and fp32) to a device input dict."""
    torch = _torch()
    dev["W_rnn"] = as_bf16_tensor(W_rnn, device)
    dev["b_rnn"] = torch.from_numpy(np.ascontiguousarray(b_rnn, dtype=np.float32)).to(device)
    return dev
