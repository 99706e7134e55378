"""Thin ctypes binding of libspecmarkov.so (see include/spec_markov.h for the semantics).

Argument marshalling only: every function here passes device pointers, sizes and the current
CUDA stream to the C entry point of the same name and allocates output tensors when the caller
does not supply them. All arithmetic of the hot path runs in the library's CUDA kernels. There is
no fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SPEC_OK = 0
SPEC_F32, SPEC_BF16 = 0, 1
(SPEC_OP_PROPOSE, SPEC_OP_VERIFY_GREEDY, SPEC_OP_VERIFY_REJECTION, SPEC_OP_TV_CONFIDENCE,
 SPEC_OP_SCHEDULE, SPEC_OP_TARGET_STATS, SPEC_OP_MTP_GREEDY, SPEC_OP_ALL) = range(8)
(SPEC_DEV_BAD_TOKEN, SPEC_DEV_NONFINITE, SPEC_DEV_EMPTY_RESIDUAL, SPEC_DEV_BAD_LENGTH,
 SPEC_DEV_TIMEOUT) = 1, 2, 4, 8, 16
SPEC_SCHEDULE_MAX_CANDIDATES = 16384
(SPEC_KCLASS_MARKOV, SPEC_KCLASS_STREAM, SPEC_KCLASS_SELECT, SPEC_KCLASS_OTHER,
 SPEC_KCLASS_PROPOSE) = range(5)
SPEC_NOALLOC_MAX_ROWS = 65536
SPEC_ERR_TOO_LARGE = -7

_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn, status):
        msg = lib().spec_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed with status {status} ({msg})")
        self.status = status


def library_path() -> str:
    return _build.SO


def lib():
    """Load libspecmarkov.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.SO):
            raise RuntimeError(f"{_build.SO} is not built; run __graft_entry__.build() first")
        L = ctypes.CDLL(_build.SO)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.spec_abi_version.restype = i
        L.spec_status_string.argtypes = [i]
        L.spec_status_string.restype = ctypes.c_char_p
        L.spec_workspace_bytes.argtypes = [i, i, i, i, i]
        L.spec_workspace_bytes.restype = sz
        L.spec_workspace_init.argtypes = [vp, sz, vp]
        L.spec_device_status.argtypes = [vp, sz, vp, ctypes.POINTER(ctypes.c_uint32), i]
        L.spec_markov_propose.argtypes = [vp, i, vp, vp, i, i, vp, vp, f, i, i, i, vp, vp, vp, vp,
                                          sz, vp]
        L.spec_verify_greedy.argtypes = [vp, i, vp, vp, i, i, i, vp, vp, vp, vp, sz, vp]
        L.spec_mtp_greedy.argtypes = [vp, vp, i, vp, i, i, i, vp, vp, vp, vp, vp, sz, vp]
        L.spec_target_stats.argtypes = [vp, i, f, i, i, vp, vp, sz, vp]
        L.spec_verify_rejection.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, vp, vp, vp, vp, vp,
                                            f, vp, i, i, i, vp, vp, vp, vp, sz, vp]
        L.spec_tv_confidence.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, vp, vp, f, i, i, i, vp,
                                         vp, vp, sz, vp]
        L.spec_schedule_prefix.argtypes = [vp, vp, i, i, i, vp, vp, vp, vp, sz, vp]
        L.spec_schedule_topk.argtypes = [vp, vp, i, i, i, vp, vp, vp, vp, vp, vp, sz, vp]
        L.spec_verify_greedy_noalloc.argtypes = [vp, i, vp, vp, i, i, i, vp, vp, vp, vp, vp]
        L.spec_markov_propose_masked.argtypes = [vp, i, vp, vp, i, i, vp, vp, f, i, i, i, vp, vp,
                                                 vp, vp, vp, sz, vp]
        L.spec_markov_propose_target_stats.argtypes = [vp, i, vp, vp, i, i, vp, vp, f, i, i, i,
                                                       vp, vp, vp, vp, vp, vp, sz, vp]
        L.spec_verify_rejection_masked.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, vp, vp, vp,
                                                   vp, vp, f, vp, i, i, i, vp, vp, vp, vp, vp,
                                                   sz, vp]
        L.spec_tv_confidence_masked.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, vp, vp, f, i, i,
                                                i, vp, vp, vp, vp, sz, vp]
        L.spec_flat_layout.argtypes = [vp, i, i, vp, vp, vp, vp, sz, vp]
        L.spec_flat_pack.argtypes = [vp, i, vp, vp, i, i, vp, vp, sz, vp]
        L.spec_target_stats_flat.argtypes = [vp, i, f, i, i, i, vp, vp, vp, sz, vp]
        L.spec_verify_greedy_flat.argtypes = [vp, i, vp, vp, vp, i, i, i, vp, vp, vp, vp, sz, vp]
        L.spec_verify_rejection_flat.argtypes = [vp, vp, i, vp, vp, i, i, vp, vp, vp, vp, vp, vp,
                                                 vp, f, vp, vp, i, i, i, vp, vp, vp, vp, vp, sz,
                                                 vp]
        L.spec_launch_count.restype = ctypes.c_ulonglong
        L.spec_trace_events.argtypes = [i, vp, vp, i]
        L.spec_trace_events.restype = i
        L.spec_trace_count.argtypes = [i]
        L.spec_trace_count.restype = i
        for name in ("spec_workspace_init", "spec_device_status", "spec_markov_propose",
                     "spec_verify_greedy", "spec_target_stats", "spec_verify_rejection",
                     "spec_tv_confidence", "spec_schedule_prefix", "spec_schedule_topk",
                     "spec_verify_greedy_noalloc", "spec_markov_propose_masked",
                     "spec_verify_rejection_masked", "spec_tv_confidence_masked",
                     "spec_markov_propose_target_stats", "spec_mtp_greedy",
                     "spec_flat_layout", "spec_flat_pack", "spec_target_stats_flat",
                     "spec_verify_greedy_flat",
                     "spec_verify_rejection_flat"):
            getattr(L, name).restype = i
        _lib = L
    return _lib


# ----------------------------------------------------------------------------- marshalling

def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits and weights must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libspecmarkov takes device tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _mask(allowed, R, V):
    """Allowed-token bitmask [R, ceil(V/32)] of 32-bit words on the device."""
    if tuple(allowed.shape) != (R, (V + 31) // 32) or allowed.element_size() != 4:
        raise ValueError(f"allowed must be [R, ceil(V/32)] = {(R, (V + 31) // 32)} 32-bit words")
    return allowed


def _check(fn, rc):
    if rc != SPEC_OK:
        raise SpecError(fn, rc)


class Workspace:
    """Caller-owned device workspace (a torch uint8 buffer) for the library's scratch."""

    def __init__(self, nbytes: int = 0, device=None):
        self.device = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        self.buf = None
        self.nbytes = 0
        if nbytes:
            self.reserve(nbytes)

    def reserve(self, nbytes: int, stream=None):
        if self.buf is not None and self.nbytes >= nbytes:
            return
        nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        base = self.buf.data_ptr()
        self._off = (-base) % 256
        self.nbytes = nbytes
        _check("spec_workspace_init", lib().spec_workspace_init(self.ptr, nbytes, _stream(stream)))

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + self._off)

    def for_op(self, op, R, gamma, V, rank, stream=None):
        self.reserve(spec_workspace_bytes(op, R, gamma, V, rank), stream)
        return self.ptr, self.nbytes

    def status(self, clear=True, stream=None) -> int:
        out = ctypes.c_uint32()
        _check("spec_device_status", lib().spec_device_status(self.ptr, self.nbytes,
                                                              _stream(stream),
                                                              ctypes.byref(out), int(clear)))
        return int(out.value)


_default_ws = {}


def default_workspace(device=None) -> Workspace:
    dev = torch.cuda.current_device() if device is None else torch.device(device).index
    if dev not in _default_ws:
        _default_ws[dev] = Workspace(device=torch.device("cuda", dev))
    return _default_ws[dev]


def spec_workspace_bytes(op, R, gamma, V, rank=0) -> int:
    return int(lib().spec_workspace_bytes(op, R, gamma, V, rank))


def spec_abi_version() -> int:
    return int(lib().spec_abi_version())


def _rank_of(W1, rank):
    if rank is not None:
        return int(rank)
    return 0 if W1 is None else int(W1.shape[1])


# ----------------------------------------------------------------------------- entry points

def spec_markov_propose(U, W1, W2, anchors, u_draft, temperature, *, rank=None,
                        draft_tokens=None, draft_logp=None, draft_stats=None, workspace=None,
                        stream=None, want_stats=True, allowed=None):
    """Draft proposal (greedy when u_draft is None or temperature == 0); `allowed` is an
    optional allowed-token bitmask [R, ceil(V/32)] (int32 / uint32 words) for grammar-masked
    drafting. Returns (draft_tokens [R,g] int32, draft_logp [R,g] fp32, draft_stats [R,g,2])."""
    R, gamma, V = U.shape
    rank = _rank_of(W1, rank)
    dev = U.device
    if draft_tokens is None:
        draft_tokens = torch.empty(R, gamma, dtype=torch.int32, device=dev)
    if want_stats and draft_logp is None:
        draft_logp = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    if want_stats and draft_stats is None:
        draft_stats = torch.empty(R, gamma, 2, dtype=torch.float32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_PROPOSE, R, gamma, V, rank, stream)
    wdt = _dt(W1) if W1 is not None else SPEC_BF16
    args = (_ptr(U), _dt(U), _ptr(W1), _ptr(W2), wdt, rank, _ptr(anchors), _ptr(u_draft),
            float(temperature), R, gamma, V, _ptr(draft_tokens), _ptr(draft_logp),
            _ptr(draft_stats))
    if allowed is None:
        rc = lib().spec_markov_propose(*args, wp, wn, _stream(stream))
    else:
        rc = lib().spec_markov_propose_masked(*args, _ptr(_mask(allowed, R, V)), wp, wn,
                                              _stream(stream))
    _check("spec_markov_propose", rc)
    return draft_tokens, draft_logp, draft_stats


def spec_markov_propose_target_stats(U, W1, W2, anchors, u_draft, temperature, target, *,
                                     rank=None, draft_tokens=None, draft_logp=None,
                                     draft_stats=None, target_stats=None, workspace=None,
                                     stream=None):
    """Draft proposal plus the target normalisers of the same window in one call. Returns
    (draft_tokens [R,g] int32, draft_logp [R,g] fp32, draft_stats [R,g,2],
    target_stats [R*(g+1), 2] fp32)."""
    R, gamma, V = U.shape
    rank = _rank_of(W1, rank)
    dev = U.device
    if draft_tokens is None:
        draft_tokens = torch.empty(R, gamma, dtype=torch.int32, device=dev)
    if draft_logp is None:
        draft_logp = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    if draft_stats is None:
        draft_stats = torch.empty(R, gamma, 2, dtype=torch.float32, device=dev)
    if target_stats is None:
        target_stats = torch.empty(R * (gamma + 1), 2, dtype=torch.float32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_PROPOSE, R, gamma, V, rank, stream)
    wdt = _dt(W1) if W1 is not None else SPEC_BF16
    rc = lib().spec_markov_propose_target_stats(
        _ptr(U), _dt(U), _ptr(W1), _ptr(W2), wdt, rank, _ptr(anchors), _ptr(u_draft),
        float(temperature), R, gamma, V, _ptr(draft_tokens), _ptr(draft_logp), _ptr(draft_stats),
        _ptr(target), _ptr(target_stats), wp, wn, _stream(stream))
    _check("spec_markov_propose_target_stats", rc)
    return draft_tokens, draft_logp, draft_stats, target_stats


def spec_mtp_greedy(D, target, lengths=None, *, draft_tokens=None, accept_len=None,
                    out_tokens=None, next_anchor=None, workspace=None, stream=None):
    """MTP/NextN greedy proposal (draft argmax per position) and greedy verification in one
    call. D [R, gamma, V] and target [R, gamma+1, V] of one dtype. Returns (draft_tokens [R,g],
    accept_len [R], out_tokens [R, g+1], next_anchor [R]), all int32."""
    R, rows, V = target.shape
    gamma = rows - 1
    dev = target.device
    if gamma > 0 and (D is None or tuple(D.shape) != (R, gamma, V) or D.dtype != target.dtype):
        raise ValueError("D must be [R, gamma, V] with the target's dtype")
    i32 = dict(dtype=torch.int32, device=dev)
    if draft_tokens is None:
        draft_tokens = torch.empty(R, gamma, **i32)
    if accept_len is None:
        accept_len = torch.empty(R, **i32)
    if out_tokens is None:
        out_tokens = torch.empty(R, gamma + 1, **i32)
    if next_anchor is None:
        next_anchor = torch.empty(R, **i32)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_MTP_GREEDY, R, gamma, V, 0, stream)
    rc = lib().spec_mtp_greedy(_ptr(D), _ptr(target), _dt(target), _ptr(lengths), R, gamma, V,
                               _ptr(draft_tokens), _ptr(accept_len), _ptr(out_tokens),
                               _ptr(next_anchor), wp, wn, _stream(stream))
    _check("spec_mtp_greedy", rc)
    return draft_tokens, accept_len, out_tokens, next_anchor


def spec_verify_greedy(target, draft_tokens, lengths=None, *, accept_len=None, out_tokens=None,
                       next_anchor=None, workspace=None, stream=None):
    R, rows, V = target.shape
    gamma = rows - 1
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(R, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R, gamma + 1, dtype=torch.int32, device=dev)
    if next_anchor is None:
        next_anchor = torch.empty(R, dtype=torch.int32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_VERIFY_GREEDY, R, gamma, V, 0, stream)
    rc = lib().spec_verify_greedy(_ptr(target), _dt(target), _ptr(draft_tokens), _ptr(lengths), R,
                                  gamma, V, _ptr(accept_len), _ptr(out_tokens), _ptr(next_anchor),
                                  wp, wn, _stream(stream))
    _check("spec_verify_greedy", rc)
    return accept_len, out_tokens, next_anchor


def spec_verify_greedy_noalloc(target, draft_tokens, lengths=None, *, accept_len=None,
                               out_tokens=None, next_anchor=None, device_status=None, stream=None):
    """spec_verify_greedy without a workspace, for callers that cannot allocate device memory
    where they call it: the library's own fixed device scratch stands in for the workspace.
    Output tensors left as None are allocated here by torch (pass them to avoid that);
    `device_status` is an optional int32 device tensor of one element that receives the call's
    SPEC_DEV_* bits."""
    R, rows, V = target.shape
    gamma = rows - 1
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(R, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R, gamma + 1, dtype=torch.int32, device=dev)
    if next_anchor is None:
        next_anchor = torch.empty(R, dtype=torch.int32, device=dev)
    rc = lib().spec_verify_greedy_noalloc(_ptr(target), _dt(target), _ptr(draft_tokens),
                                          _ptr(lengths), R, gamma, V, _ptr(accept_len),
                                          _ptr(out_tokens), _ptr(next_anchor),
                                          _ptr(device_status), _stream(stream))
    _check("spec_verify_greedy_noalloc", rc)
    return accept_len, out_tokens, next_anchor


def spec_target_stats(target, temperature, *, stats=None, workspace=None, stream=None):
    V = target.shape[-1]
    rows = target.numel() // V
    if stats is None:
        stats = torch.empty(rows, 2, dtype=torch.float32, device=target.device)
    ws = workspace or default_workspace(target.device)
    wp, wn = ws.for_op(SPEC_OP_TARGET_STATS, 1 if rows else 0, max(rows - 1, 0), V, 0, stream)
    rc = lib().spec_target_stats(_ptr(target), _dt(target), float(temperature), rows, V,
                                 _ptr(stats), wp, wn, _stream(stream))
    _check("spec_target_stats", rc)
    return stats


def spec_verify_rejection(target, U, W1, W2, anchors, draft_tokens, draft_logp, draft_stats,
                          u_accept, u_resid, temperature, lengths=None, *, rank=None,
                          target_stats=None, accept_len=None, out_tokens=None, next_anchor=None,
                          workspace=None, stream=None, allowed=None):
    R, gamma, V = U.shape
    rank = _rank_of(W1, rank)
    dev = U.device
    if accept_len is None:
        accept_len = torch.empty(R, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R, gamma + 1, dtype=torch.int32, device=dev)
    if next_anchor is None:
        next_anchor = torch.empty(R, dtype=torch.int32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_VERIFY_REJECTION, R, gamma, V, rank, stream)
    wdt = _dt(W1) if W1 is not None else SPEC_BF16
    args = (_ptr(target), _ptr(U), _dt(U), _ptr(W1), _ptr(W2), wdt, rank, _ptr(anchors),
            _ptr(draft_tokens), _ptr(draft_logp), _ptr(draft_stats), _ptr(target_stats),
            _ptr(u_accept), _ptr(u_resid), float(temperature), _ptr(lengths), R, gamma, V,
            _ptr(accept_len), _ptr(out_tokens), _ptr(next_anchor))
    if allowed is None:
        rc = lib().spec_verify_rejection(*args, wp, wn, _stream(stream))
    else:
        rc = lib().spec_verify_rejection_masked(*args, _ptr(_mask(allowed, R, V)), wp, wn,
                                                _stream(stream))
    _check("spec_verify_rejection", rc)
    return accept_len, out_tokens, next_anchor


def spec_tv_confidence(U, target, W1, W2, anchors, draft_tokens, temperature, *, rank=None,
                       draft_stats=None, target_stats=None, conf=None, survival=None,
                       workspace=None, stream=None, allowed=None):
    R, gamma, V = U.shape
    rank = _rank_of(W1, rank)
    dev = U.device
    if conf is None:
        conf = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    if survival is None:
        survival = torch.empty(R, gamma, dtype=torch.float32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_TV_CONFIDENCE, R, gamma, V, rank, stream)
    wdt = _dt(W1) if W1 is not None else SPEC_BF16
    args = (_ptr(U), _ptr(target), _dt(U), _ptr(W1), _ptr(W2), wdt, rank, _ptr(anchors),
            _ptr(draft_tokens), _ptr(draft_stats), _ptr(target_stats), float(temperature), R,
            gamma, V, _ptr(conf), _ptr(survival))
    if allowed is None:
        rc = lib().spec_tv_confidence(*args, wp, wn, _stream(stream))
    else:
        rc = lib().spec_tv_confidence_masked(*args, _ptr(_mask(allowed, R, V)), wp, wn,
                                             _stream(stream))
    _check("spec_tv_confidence", rc)
    return conf, survival


def spec_schedule_prefix(survival, sps, *, lengths=None, B_out=None, theta_out=None,
                         workspace=None, stream=None, capacity=None, B_opt_out=None):
    """Prefix scheduler. With `capacity` (a [1] int32 device tensor holding a batch size,
    typically the Theta-optimal batch of an earlier step) it is the dynamic top-K selection
    instead of the Theta search; `B_opt_out` ([1] int32, optional) then receives this step's
    Theta-optimal batch size."""
    R, gamma = survival.shape
    dev = survival.device
    if lengths is None:
        lengths = torch.empty(R, dtype=torch.int32, device=dev)
    if B_out is None:
        B_out = torch.empty(1, dtype=torch.int32, device=dev)
    if theta_out is None:
        theta_out = torch.empty(1, dtype=torch.float64, device=dev)
    ws = workspace or default_workspace(dev)
    ws.reserve(256, stream)
    if capacity is None:
        if B_opt_out is not None:
            raise ValueError("B_opt_out is an output of the capacity form")
        rc = lib().spec_schedule_prefix(_ptr(survival), _ptr(sps), sps.numel() - 1, R, gamma,
                                        _ptr(lengths), _ptr(B_out), _ptr(theta_out), ws.ptr,
                                        ws.nbytes, _stream(stream))
    else:
        if capacity.dtype != torch.int32 or capacity.numel() < 1 or capacity.device != dev:
            raise ValueError("capacity must be an int32 tensor on the survival's device")
        if B_opt_out is not None and (B_opt_out.dtype != torch.int32 or B_opt_out.device != dev):
            raise ValueError("B_opt_out must be an int32 tensor on the survival's device")
        rc = lib().spec_schedule_topk(_ptr(survival), _ptr(sps), sps.numel() - 1, R, gamma,
                                      _ptr(capacity), _ptr(lengths), _ptr(B_out),
                                      _ptr(theta_out),
                                      None if B_opt_out is None else _ptr(B_opt_out), ws.ptr,
                                      ws.nbytes, _stream(stream))
    _check("spec_schedule_prefix", rc)
    return lengths, B_out, theta_out


# ----------------------------------------------------------------------------- flattened batch

def _i32_on(t, dev, name):
    if t.dtype != torch.int32 or t.device != dev:
        raise ValueError(f"{name} must be an int32 tensor on {dev}")
    return t


def spec_flat_layout(lengths, gamma, *, offsets=None, row_req=None, row_pos=None, markers=True,
                     workspace=None, stream=None):
    """Packed-row layout of a variable-length verify batch: offsets [R+1] (offsets[R] = B) and,
    with markers=True, the request / position of each of the R*(gamma+1) packed rows (-1 past
    B). Returns (offsets, row_req, row_pos)."""
    R = lengths.shape[0]
    dev = lengths.device
    _i32_on(lengths, dev, "lengths")
    if offsets is None:
        offsets = torch.empty(R + 1, dtype=torch.int32, device=dev)
    if markers and row_req is None:
        row_req = torch.empty(R * (gamma + 1), dtype=torch.int32, device=dev)
    if markers and row_pos is None:
        row_pos = torch.empty(R * (gamma + 1), dtype=torch.int32, device=dev)
    ws = workspace or default_workspace(dev)
    ws.reserve(256, stream)
    rc = lib().spec_flat_layout(_ptr(lengths), R, int(gamma), _ptr(offsets), _ptr(row_req),
                                _ptr(row_pos), ws.ptr, ws.nbytes, _stream(stream))
    _check("spec_flat_layout", rc)
    return offsets, row_req, row_pos


def spec_flat_pack(src, lengths, offsets, *, out=None, workspace=None, stream=None):
    """Rows (r, i <= l_r) of a padded src [R, gamma+1, ...] to packed rows offsets[r] + i of
    out [R*(gamma+1), ...] (allocated when None; rows past B are left as they were)."""
    R, g1 = src.shape[0], src.shape[1]
    dev = src.device
    _i32_on(lengths, dev, "lengths")
    _i32_on(offsets, dev, "offsets")
    row_bytes = src[0, 0].numel() * src.element_size() if src.numel() else 4
    if out is None:
        out = torch.empty((R * g1,) + tuple(src.shape[2:]), dtype=src.dtype, device=dev)
    if out.numel() != src.numel() or out.dtype != src.dtype:
        raise ValueError("out holds R*(gamma+1) rows of src's row shape and dtype")
    ws = workspace or default_workspace(dev)
    ws.reserve(256, stream)
    rc = lib().spec_flat_pack(_ptr(src), int(row_bytes), _ptr(lengths), _ptr(offsets), R,
                              g1 - 1, _ptr(out), ws.ptr, ws.nbytes, _stream(stream))
    _check("spec_flat_pack", rc)
    return out


def spec_target_stats_flat(target, temperature, offsets, gamma, *, stats=None, workspace=None,
                           stream=None):
    """(m, log Z) of the packed target rows b < offsets[R]; target [R*(gamma+1), V]."""
    R = offsets.shape[0] - 1
    V = target.shape[-1]
    dev = target.device
    if target.numel() != R * (gamma + 1) * V:
        raise ValueError("a packed target holds R*(gamma+1) rows")
    _i32_on(offsets, dev, "offsets")
    if stats is None:
        stats = torch.empty(R * (gamma + 1), 2, dtype=torch.float32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_TARGET_STATS, R, gamma, V, 0, stream)
    rc = lib().spec_target_stats_flat(_ptr(target), _dt(target), float(temperature), R,
                                      int(gamma), V, _ptr(offsets), _ptr(stats), wp, wn,
                                      _stream(stream))
    _check("spec_target_stats_flat", rc)
    return stats


def spec_verify_greedy_flat(target, draft_tokens, lengths, offsets, *, accept_len=None,
                            out_tokens=None, next_anchor=None, workspace=None, stream=None):
    """Greedy verify with the target rows packed by spec_flat_layout (target [R*(gamma+1), V])."""
    R, gamma = draft_tokens.shape
    V = target.shape[-1]
    dev = target.device
    if target.numel() != R * (gamma + 1) * V:
        raise ValueError("a packed target holds R*(gamma+1) rows")
    _i32_on(lengths, dev, "lengths")
    _i32_on(offsets, dev, "offsets")
    if accept_len is None:
        accept_len = torch.empty(R, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R, gamma + 1, dtype=torch.int32, device=dev)
    if next_anchor is None:
        next_anchor = torch.empty(R, dtype=torch.int32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_VERIFY_GREEDY, R, gamma, V, 0, stream)
    rc = lib().spec_verify_greedy_flat(_ptr(target), _dt(target), _ptr(draft_tokens),
                                       _ptr(lengths), _ptr(offsets), R, gamma, V,
                                       _ptr(accept_len), _ptr(out_tokens), _ptr(next_anchor),
                                       wp, wn, _stream(stream))
    _check("spec_verify_greedy_flat", rc)
    return accept_len, out_tokens, next_anchor


def spec_verify_rejection_flat(target, U, W1, W2, anchors, draft_tokens, draft_logp,
                               draft_stats, u_accept, u_resid, temperature, lengths, offsets, *,
                               rank=None, target_stats=None, accept_len=None, out_tokens=None,
                               next_anchor=None, workspace=None, stream=None, allowed=None):
    """Rejection verify with the target rows (and target_stats, if given) packed by
    spec_flat_layout; everything else keeps its per-request layout."""
    R, gamma, V = U.shape
    rank = _rank_of(W1, rank)
    dev = U.device
    if target.numel() != R * (gamma + 1) * V:
        raise ValueError("a packed target holds R*(gamma+1) rows")
    _i32_on(lengths, dev, "lengths")
    _i32_on(offsets, dev, "offsets")
    if accept_len is None:
        accept_len = torch.empty(R, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R, gamma + 1, dtype=torch.int32, device=dev)
    if next_anchor is None:
        next_anchor = torch.empty(R, dtype=torch.int32, device=dev)
    ws = workspace or default_workspace(dev)
    wp, wn = ws.for_op(SPEC_OP_VERIFY_REJECTION, R, gamma, V, rank, stream)
    wdt = _dt(W1) if W1 is not None else SPEC_BF16
    mask = None if allowed is None else _mask(allowed, R, V)
    rc = lib().spec_verify_rejection_flat(
        _ptr(target), _ptr(U), _dt(U), _ptr(W1), _ptr(W2), wdt, rank, _ptr(anchors),
        _ptr(draft_tokens), _ptr(draft_logp), _ptr(draft_stats), _ptr(target_stats),
        _ptr(u_accept), _ptr(u_resid), float(temperature), _ptr(lengths), _ptr(offsets), R,
        gamma, V, _ptr(accept_len), _ptr(out_tokens), _ptr(next_anchor), _ptr(mask), wp, wn,
        _stream(stream))
    _check("spec_verify_rejection_flat", rc)
    return accept_len, out_tokens, next_anchor


def spec_device_status(workspace=None, clear=True, stream=None) -> int:
    ws = workspace or default_workspace()
    return ws.status(clear=clear, stream=stream)
