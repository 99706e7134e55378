"""CPU oracle for the speculative-decoding hot path (test infrastructure only).

The oracle is `spec_oracle.c`, a plain C restatement of what the pages define (see the header
comment of that file for every passage and reading). This module builds it with gcc and
exposes it through ctypes with numpy arrays.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. The product library never does.

Array conventions (all C-contiguous, host memory):
  * logits / weights: ``float32`` arrays, or ``uint16`` arrays holding raw bfloat16 bits
    (numpy has no bfloat16); torch tensors of either dtype are accepted and converted.
  * token ids: ``int32``; uniforms: ``float32``; probabilities and margins come back as
    ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

F32, BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_lib")
_SO = os.path.join(_LIB_DIR, "libspec_oracle.so")

_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into a shared library (gcc, fp contraction off, OpenMP)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        c_i32p = ctypes.POINTER(ctypes.c_int32)
        c_dp = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        i = ctypes.c_int
        f = ctypes.c_float
        lib.oracle_num_threads.restype = i
        lib.oracle_softmax.argtypes = [c_dp, i, c_dp, c_dp, c_dp]
        lib.oracle_softmax.restype = None
        lib.oracle_argmax.argtypes = [c_dp, i, c_dp]
        lib.oracle_argmax.restype = i
        lib.oracle_sample.argtypes = [c_dp, i, ctypes.c_double, c_dp]
        lib.oracle_sample.restype = i
        lib.oracle_accept_test.argtypes = [ctypes.c_double] * 3
        lib.oracle_accept_test.restype = i
        lib.oracle_accept_prob.argtypes = [ctypes.c_double] * 2
        lib.oracle_accept_prob.restype = ctypes.c_double
        lib.oracle_residual.argtypes = [c_dp, c_dp, i, c_dp]
        lib.oracle_residual.restype = ctypes.c_double
        lib.oracle_draft_probs.argtypes = [vp, i, vp, vp, i, i, i, i, i, i, i, ctypes.c_int32,
                                           f, c_dp, c_dp, c_dp, vp]
        lib.oracle_draft_probs.restype = i
        lib.oracle_target_probs.argtypes = [vp, i, i, i, i, i, i, f, c_dp]
        lib.oracle_target_probs.restype = i
        lib.oracle_markov_propose.argtypes = [vp, i, vp, vp, i, i, vp, vp, f, i, i, i, vp, vp, vp,
                                              vp, vp]
        lib.oracle_markov_propose.restype = i
        lib.oracle_verify_greedy.argtypes = [vp, i, vp, vp, i, i, i, vp, vp, vp]
        lib.oracle_verify_greedy.restype = i
        lib.oracle_verify_rejection.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, vp, vp, f, vp, i,
                                                i, i, vp, vp, vp, vp, vp, vp]
        lib.oracle_verify_rejection.restype = i
        lib.oracle_tv_confidence.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, f, i, i, i, vp, vp,
                                             vp]
        lib.oracle_tv_confidence.restype = i
        lib.oracle_schedule_prefix.argtypes = [vp, vp, i, i, i, vp, vp, vp]
        lib.oracle_schedule_prefix.restype = i
        lib.oracle_schedule_topk.argtypes = [vp, vp, i, i, i, i, vp, vp, vp]
        lib.oracle_schedule_topk.restype = i
        lib.oracle_flat_layout.argtypes = [vp, i, i, vp, vp, vp]
        lib.oracle_flat_layout.restype = i
        del c_i32p
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------------------- marshalling

def _np(a):
    """torch tensor or numpy array -> C-contiguous numpy array (bf16 -> uint16 raw bits)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            t = a.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a)


def _logits(a):
    a = _np(a)
    if a is None:
        return None, F32
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"logits/weights must be float32 or raw bf16 (uint16), got {a.dtype}")


def _i32(a):
    a = _np(a)
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _f32(a):
    a = _np(a)
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _mask(a, R, V):
    """Allowed-token bitmask [R, ceil(V/32)] as uint32 words, or None."""
    a = _np(a)
    if a is None:
        return None
    a = np.ascontiguousarray(a).view(np.uint32) if a.dtype.itemsize == 4 else a
    a = np.ascontiguousarray(a, dtype=np.uint32)
    if a.shape != (R, (V + 31) // 32):
        raise ValueError(f"mask must be [R, ceil(V/32)] = {(R, (V + 31) // 32)}, got {a.shape}")
    return a


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} returned status {rc}")


# ----------------------------------------------------------------------------- building blocks

def softmax(z):
    z = np.ascontiguousarray(z, dtype=np.float64)
    p = np.empty_like(z)
    m = ctypes.c_double()
    lz = ctypes.c_double()
    _load().oracle_softmax(_dp(z), z.size, _dp(p), ctypes.byref(m), ctypes.byref(lz))
    return p, m.value, lz.value


def argmax(s):
    s = np.ascontiguousarray(s, dtype=np.float64)
    gap = ctypes.c_double()
    v = _load().oracle_argmax(_dp(s), s.size, ctypes.byref(gap))
    return int(v), gap.value


def sample(p, u):
    p = np.ascontiguousarray(p, dtype=np.float64)
    mrg = ctypes.c_double()
    v = _load().oracle_sample(_dp(p), p.size, float(u), ctypes.byref(mrg))
    return int(v), mrg.value


def accept_test(u, pd_x, pt_x) -> bool:
    return bool(_load().oracle_accept_test(float(u), float(pd_x), float(pt_x)))


def accept_prob(pd_x, pt_x) -> float:
    return float(_load().oracle_accept_prob(float(pd_x), float(pt_x)))


def residual(pt, pd):
    pt = np.ascontiguousarray(pt, dtype=np.float64)
    pd = np.ascontiguousarray(pd, dtype=np.float64)
    q = np.empty_like(pt)
    z = _load().oracle_residual(_dp(pt), _dp(pd), pt.size, _dp(q))
    return q, float(z)


def draft_probs(U, W1, W2, r, k, prev, temperature, rank=None, mask=None):
    """p_d at draft position k (1-based) of request r after token prev (mask: allowed-token
    bitmask [R, ceil(V/32)] or None)."""
    U, ud = _logits(U)
    W1, wd = _logits(W1)
    W2, _ = _logits(W2)
    R, gamma, V = U.shape
    rank = (W1.shape[1] if W1 is not None else 0) if rank is None else rank
    p = np.empty(V, dtype=np.float64)
    m = ctypes.c_double()
    lz = ctypes.c_double()
    rc = _load().oracle_draft_probs(_p(U), ud, _p(W1), _p(W2), wd, rank, R, gamma, V, r, k,
                                    int(prev), float(temperature), _dp(p), ctypes.byref(m),
                                    ctypes.byref(lz), _p(_mask(mask, R, V)))
    _check(rc, "oracle_draft_probs")
    return p, m.value, lz.value


def target_probs(target, r, i, temperature):
    T, td = _logits(target)
    R, rows, V = T.shape
    p = np.empty(V, dtype=np.float64)
    rc = _load().oracle_target_probs(_p(T), td, R, rows, V, r, i, float(temperature), _dp(p))
    _check(rc, "oracle_target_probs")
    return p


# ----------------------------------------------------------------------------- the five steps

def markov_propose(U, W1, W2, anchors, u_draft, temperature, rank=None, mask=None):
    """Draft proposal. Returns dict(tokens [R,g] i32, logp [R,g], stats [R,g,2], margin [R,g])."""
    U, ud = _logits(U)
    W1, wd = _logits(W1)
    W2, wd2 = _logits(W2)
    if W1 is not None and wd != wd2:
        raise TypeError("W1 and W2 must share a dtype")
    R, gamma, V = U.shape
    rank = (W1.shape[1] if W1 is not None else 0) if rank is None else rank
    anchors = _i32(anchors)
    u_draft = _f32(u_draft)
    tokens = np.empty((R, gamma), dtype=np.int32)
    logp = np.empty((R, gamma), dtype=np.float64)
    stats = np.empty((R, gamma, 2), dtype=np.float64)
    margin = np.empty((R, gamma), dtype=np.float64)
    rc = _load().oracle_markov_propose(_p(U), ud, _p(W1), _p(W2), wd, rank, _p(anchors),
                                       _p(u_draft), float(temperature), R, gamma, V, _p(tokens),
                                       _p(logp), _p(stats), _p(margin), _p(_mask(mask, R, V)))
    _check(rc, "oracle_markov_propose")
    return dict(tokens=tokens, logp=logp, stats=stats, margin=margin)


def verify_greedy(target, draft_tokens, lengths=None):
    T, td = _logits(target)
    R, rows, V = T.shape
    gamma = rows - 1
    draft_tokens = _i32(draft_tokens)
    lengths = _i32(lengths)
    n = np.empty(R, dtype=np.int32)
    out = np.empty((R, gamma + 1), dtype=np.int32)
    nxt = np.empty(R, dtype=np.int32)
    rc = _load().oracle_verify_greedy(_p(T), td, _p(draft_tokens), _p(lengths), R, gamma, V,
                                      _p(n), _p(out), _p(nxt))
    _check(rc, "oracle_verify_greedy")
    return dict(accept_len=n, out_tokens=out, next_anchor=nxt)


def verify_rejection(target, U, W1, W2, anchors, draft_tokens, u_accept, u_resid, temperature,
                     lengths=None, rank=None, mask=None):
    T, td = _logits(target)
    U, ud = _logits(U)
    if td != ud:
        raise TypeError("target and U must share a dtype")
    W1, wd = _logits(W1)
    W2, _ = _logits(W2)
    R, gamma, V = U.shape
    rank = (W1.shape[1] if W1 is not None else 0) if rank is None else rank
    n = np.empty(R, dtype=np.int32)
    out = np.empty((R, gamma + 1), dtype=np.int32)
    nxt = np.empty(R, dtype=np.int32)
    am = np.empty((R, gamma), dtype=np.float64)
    rm = np.empty(R, dtype=np.float64)
    rc = _load().oracle_verify_rejection(_p(T), _p(U), td, _p(W1), _p(W2), wd, rank,
                                         _p(_i32(anchors)), _p(_i32(draft_tokens)),
                                         _p(_f32(u_accept)), _p(_f32(u_resid)),
                                         float(temperature), _p(_i32(lengths)), R, gamma, V,
                                         _p(n), _p(out), _p(nxt), _p(am), _p(rm),
                                         _p(_mask(mask, R, V)))
    _check(rc, "oracle_verify_rejection")
    return dict(accept_len=n, out_tokens=out, next_anchor=nxt, accept_margin=am,
                resid_margin=rm)


def tv_confidence(U, target, W1, W2, anchors, draft_tokens, temperature, rank=None, mask=None):
    U, ud = _logits(U)
    T, td = _logits(target)
    if td != ud:
        raise TypeError("target and U must share a dtype")
    W1, wd = _logits(W1)
    W2, _ = _logits(W2)
    R, gamma, V = U.shape
    rank = (W1.shape[1] if W1 is not None else 0) if rank is None else rank
    conf = np.empty((R, gamma), dtype=np.float64)
    surv = np.empty((R, gamma), dtype=np.float64)
    rc = _load().oracle_tv_confidence(_p(U), _p(T), ud, _p(W1), _p(W2), wd, rank,
                                      _p(_i32(anchors)), _p(_i32(draft_tokens)),
                                      float(temperature), R, gamma, V, _p(conf), _p(surv),
                                      _p(_mask(mask, R, V)))
    _check(rc, "oracle_tv_confidence")
    return dict(conf=conf, survival=surv)


def schedule_prefix(survival, sps):
    a = _f32(survival)
    R, gamma = a.shape
    sps = np.ascontiguousarray(sps, dtype=np.float64)
    lengths = np.empty(R, dtype=np.int32)
    B = ctypes.c_int32()
    theta = ctypes.c_double()
    rc = _load().oracle_schedule_prefix(_p(a), _p(sps), sps.size - 1, R, gamma, _p(lengths),
                                        ctypes.cast(ctypes.byref(B), ctypes.c_void_p),
                                        ctypes.cast(ctypes.byref(theta), ctypes.c_void_p))
    _check(rc, "oracle_schedule_prefix")
    return dict(lengths=lengths, B=int(B.value), theta=float(theta.value))


def schedule_topk(survival, sps, capacity):
    """Dynamic top-K (DSpark section 7): the batch size `capacity` is given (from an earlier
    step's confidences); the first K = capacity - R candidates of the current queue are taken."""
    a = _f32(survival)
    R, gamma = a.shape
    sps = np.ascontiguousarray(sps, dtype=np.float64)
    lengths = np.empty(R, dtype=np.int32)
    B = ctypes.c_int32()
    theta = ctypes.c_double()
    rc = _load().oracle_schedule_topk(_p(a), _p(sps), sps.size - 1, R, gamma, int(capacity),
                                      _p(lengths), ctypes.cast(ctypes.byref(B), ctypes.c_void_p),
                                      ctypes.cast(ctypes.byref(theta), ctypes.c_void_p))
    _check(rc, "oracle_schedule_topk")
    return dict(lengths=lengths, B=int(B.value), theta=float(theta.value))


def flat_layout(lengths, gamma):
    """Packed-row layout of a variable-length verify batch (DSpark section 7): offsets [R+1],
    and the request / position of each of the R*(gamma+1) packed rows (-1 past the batch)."""
    ln = _i32(lengths)
    R = ln.shape[0]
    offsets = np.empty(R + 1, dtype=np.int32)
    row_req = np.empty(R * (gamma + 1), dtype=np.int32)
    row_pos = np.empty(R * (gamma + 1), dtype=np.int32)
    _check(_load().oracle_flat_layout(_p(ln), R, int(gamma), _p(offsets), _p(row_req),
                                      _p(row_pos)), "oracle_flat_layout")
    return dict(offsets=offsets, row_req=row_req, row_pos=row_pos)
