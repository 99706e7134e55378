"""spec_verify_greedy_noalloc: greedy verification for callers that cannot allocate device memory
at the call site (an engine plug-in whose device memory is all reserved at start-up, a loop that
must not meet cudaMalloc's implicit synchronisation). Its scratch is a fixed array inside the
library instead of a caller workspace, so it must give exactly what spec_verify_greedy gives,
call after call, although each call inherits the array as the previous call left it.

The file name sorts last so that a run stopping at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from draft_sampling_verification_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SPEC_DEV_BAD_LENGTH = 0x8


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def _noalloc(spec, target, tokens, lengths):
    """One call of the C entry point; outputs and the status slot are made beforehand."""
    R, rows, V = target.shape
    dev = target.device
    n = torch.full((R,), -7, dtype=torch.int32, device=dev)
    out = torch.full((R, rows), -7, dtype=torch.int32, device=dev)
    nxt = torch.full((R,), -7, dtype=torch.int32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    vp = ctypes.c_void_p
    rc = spec.lib().spec_verify_greedy_noalloc(
        vp(target.data_ptr()), spec.SPEC_BF16 if target.dtype == torch.bfloat16 else spec.SPEC_F32,
        vp(tokens.data_ptr()), None if lengths is None else vp(lengths.data_ptr()), R, rows - 1, V,
        vp(n.data_ptr()), vp(out.data_ptr()), vp(nxt.data_ptr()), vp(status.data_ptr()),
        vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, spec.lib().spec_status_string(rc)
    return n, out, nxt, status


def _with_workspace(spec, target, tokens, lengths):
    ws = spec.Workspace(device="cuda")
    n, out, nxt = spec.spec_verify_greedy(target, tokens, lengths, workspace=ws)
    torch.cuda.synchronize()
    return n, out, nxt, ws.status()


def _same(a, b):
    # integer outputs: the tolerance is exact equality
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(spec):
    # call 1: bf16 MTP-style window, full vocabulary, one request with a length outside
    # [0, gamma] so that the call leaves a status bit behind in the shared scratch
    big = W.mtp_greedy("cuda", R=64, gamma=3, V=129280, seed=21)
    tokens = big.extra["planted_tokens"].cuda()
    lengths = torch.tensor([i % 4 for i in range(64)], dtype=torch.int32, device="cuda")
    lengths[5] = 9
    first = _noalloc(spec, big.target, tokens, lengths)
    torch.cuda.synchronize()
    ref = _with_workspace(spec, big.target, tokens, lengths)
    _same(first, ref)
    assert first[3].item() == SPEC_DEV_BAD_LENGTH == ref[3]

    # call 2, straight after: a smaller fp32 problem with a ragged vocabulary; the argmax rows
    # and the status word left by call 1 must not show through
    small = W.greedy_toy("cuda", R=5, gamma=4, V=1003, rank=16, seed=22)
    toks = torch.randint(0, 1003, (5, 4), dtype=torch.int32, device="cuda")
    toks[:, 0] = small.target[:, 0, :].argmax(-1).to(torch.int32)  # some prefixes survive
    second = _noalloc(spec, small.target, toks, None)
    torch.cuda.synchronize()
    ref2 = _with_workspace(spec, small.target, toks, None)
    _same(second, ref2)
    assert second[3].item() == 0 == ref2[3]
    assert (second[0] >= 1).all()


def test_noalloc_rejects_sizes_beyond_its_scratch(spec):
    R = spec.SPEC_NOALLOC_MAX_ROWS // 4 + 1  # R * (gamma + 1) one request past the limit
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    before = spec.lib().spec_launch_count()
    rc = spec.lib().spec_verify_greedy_noalloc(p, spec.SPEC_F32, p, None, R, 3, 8, p, p, p, None,
                                               None)
    assert rc == spec.SPEC_ERR_TOO_LARGE
    assert b"fixed scratch" in spec.lib().spec_status_string(rc)
    assert spec.lib().spec_launch_count() == before
