"""Failure detection on the GPU without a fault: every wait of the tensor-core Markov kernel is
bounded. A test hook makes one wait run out (the first W2 tile of the next Markov pass is never
loaded); the kernel must report SPEC_DEV_TIMEOUT through the device status word, return, and
leave the CUDA context usable, so that the next call gives correct results."""
import time

import pytest
import torch

from draft_sampling_verification_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SPEC_DEV_TIMEOUT = 0x10


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def test_expired_wait_reports_timeout_and_context_survives(spec):
    wl = W.markov_rejection("cuda", R=130, gamma=2, V=4096, rank=128, seed=41)
    run = lambda ws: spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, None, 0.0,
                                              workspace=ws)
    ref_ws = spec.Workspace(device="cuda")
    ref = [x.clone() for x in run(ref_ws)]
    torch.cuda.synchronize()
    assert ref_ws.status() == 0

    ws = spec.Workspace(device="cuda")
    run(ws)                              # sizes the workspace
    torch.cuda.synchronize()
    assert spec.lib().spec_test_stall_next_markov() == 0
    t0 = time.time()
    run(ws)                              # position 1's Markov pass waits in vain, then returns
    torch.cuda.synchronize()             # no CUDA error: the kernels completed
    waited = time.time() - t0
    status = ws.status(clear=True)
    assert status & SPEC_DEV_TIMEOUT, f"status {status:#x}"
    assert 0.5 < waited < 30.0

    again = run(ws)                      # the context and the workspace are usable
    torch.cuda.synchronize()
    assert ws.status() == 0
    for a, b in zip(again, ref):
        assert torch.equal(a, b)


def test_expired_wait_in_the_fused_launch(spec):
    """The same with the target normalisers in the launch (statistics CTAs beside the
    proposal): the stalled launch reports SPEC_DEV_TIMEOUT and returns, and the next call gives
    the proposal and the normalisers of an unstalled run."""
    wl = W.markov_rejection("cuda", R=130, gamma=2, V=4096, rank=128, seed=42)
    run = lambda ws: spec.spec_markov_propose_target_stats(wl.U, wl.W1, wl.W2, wl.anchors, None,
                                                           1.0, wl.target, workspace=ws)
    ref_ws = spec.Workspace(device="cuda")
    ref = [x.clone() for x in run(ref_ws)]
    torch.cuda.synchronize()
    assert ref_ws.status() == 0

    ws = spec.Workspace(device="cuda")
    run(ws)
    torch.cuda.synchronize()
    assert spec.lib().spec_test_stall_next_markov() == 0
    t0 = time.time()
    run(ws)
    torch.cuda.synchronize()
    waited = time.time() - t0
    status = ws.status(clear=True)
    assert status & SPEC_DEV_TIMEOUT, f"status {status:#x}"
    assert 0.5 < waited < 30.0

    again = run(ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    for a, b in zip(again, ref):
        assert torch.equal(a, b)


def test_expired_wait_in_the_residual_pass(spec):
    """The same on the residual pass of rejection verification (gathered final rows, six copier
    warps and a register split between warpgroups): the stalled pass reports SPEC_DEV_TIMEOUT
    and returns, and the next verify gives the results of an unstalled run."""
    wl = W.markov_rejection("cuda", R=130, gamma=3, V=4096, rank=128, seed=43)
    ws = spec.Workspace(device="cuda")
    toks, logp, stats = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft,
                                                 1.0, workspace=ws)
    tst = spec.spec_target_stats(wl.target, 1.0, workspace=ws)
    ver = lambda: spec.spec_verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, toks,
                                             logp, stats, wl.u_accept, wl.u_resid, 1.0,
                                             target_stats=tst, workspace=ws)
    ref = [x.clone() for x in ver()]
    torch.cuda.synchronize()
    assert ws.status() == 0

    assert spec.lib().spec_test_stall_next_markov() == 0
    t0 = time.time()
    ver()
    torch.cuda.synchronize()
    waited = time.time() - t0
    status = ws.status(clear=True)
    assert status & SPEC_DEV_TIMEOUT, f"status {status:#x}"
    assert 0.5 < waited < 30.0

    again = ver()
    torch.cuda.synchronize()
    assert ws.status() == 0
    for a, b in zip(again, ref):
        assert torch.equal(a, b)
