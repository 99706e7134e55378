"""Parity at the full sizes of the workloads (the benchmarked one in the launch configuration
bench.py times): the whole batch runs on the GPU; the oracle recomputes a sample of requests
one by one (requests are independent in proposal and verification), and properties that hold
at any size are checked on every request."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import assert_conf_close, compare_proposals
from test_gpu_loop import check_iteration

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def test_markov_rejection_full_size_sampled(spec):
    R, g, V = 256, 7, 129280
    wl = W.markov_rejection("cuda", R=R, gamma=g, V=V, rank=256, seed=1003)
    ws = spec.Workspace(device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        toks, logp, stats = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft,
                                                     1.0, workspace=ws, stream=stream)
        tst = spec.spec_target_stats(wl.target, 1.0, workspace=ws, stream=stream)
        n, out, nxt = spec.spec_verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, toks,
                                                 logp, stats, wl.u_accept, wl.u_resid, 1.0,
                                                 target_stats=tst, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    assert ws.status() == 0
    # properties on every request
    t, nn, o = toks.cpu().numpy(), n.cpu().numpy(), out.cpu().numpy()
    assert ((t >= 0) & (t < V)).all()
    assert ((nn >= 0) & (nn <= g)).all()
    for r in range(R):
        assert (o[r, :nn[r]] == t[r, :nn[r]]).all() and 0 <= o[r, nn[r]] < V
        assert (o[r, nn[r] + 1:] == -1).all()
    np.testing.assert_array_equal(nxt.cpu().numpy(), o[np.arange(R), nn])
    # oracle on a sample of requests (first, last, and a few inside; two 128-row tiles)
    sample = [0, 1, 127, 128, 200, 255]
    sl = lambda x: x[sample].cpu()
    ref = oracle.markov_propose(sl(wl.U), wl.W1.cpu(), wl.W2.cpu(), sl(wl.anchors),
                                sl(wl.u_draft), 1.0)
    same = compare_proposals(toks[sample], logp[sample], stats[sample], ref)
    rv = oracle.verify_rejection(sl(wl.target), sl(wl.U), wl.W1.cpu(), wl.W2.cpu(),
                                 sl(wl.anchors), ref["tokens"], sl(wl.u_accept), sl(wl.u_resid),
                                 1.0)
    amb = (np.nan_to_num(rv["accept_margin"], nan=1.0) < 1e-6).any(axis=1) | (
        rv["resid_margin"] < 1e-6)
    for si, r in enumerate(sample):
        if same[si] and not amb[si]:
            assert nn[r] == rv["accept_len"][si]
            np.testing.assert_array_equal(o[r], rv["out_tokens"][si])
    # target normalisers of the sampled requests' rows
    st = tst.cpu().numpy().reshape(R, g + 1, 2)
    for si, r in enumerate(sample[:2]):
        for i in range(g + 1):
            z = wl.target[r, i].double().cpu().numpy()
            m = z.max()
            lz = np.log(np.exp(z - m).sum())
            assert abs((st[r, i, 0] + st[r, i, 1]) - (m + lz)) <= 1e-5 * max(1, abs(m + lz))


def test_confidence_scheduling_full_size_sampled(spec):
    """R = 512, gamma = 16: proposal, target normalisers, TV confidence with survival, and the
    scheduler over all 8192 candidates (bit-exact on the GPU's survival)."""
    R, g, V = 512, 16, 129280
    wl = W.confidence_scheduling("cuda", R=R, gamma=g, V=V, rank=256, seed=1004)
    ws = spec.Workspace(device="cuda")
    toks, logp, stats = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, 1.0,
                                                 workspace=ws)
    tst = spec.spec_target_stats(wl.target, 1.0, workspace=ws)
    conf, surv = spec.spec_tv_confidence(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, toks, 1.0,
                                         draft_stats=stats, target_stats=tst, workspace=ws)
    sps = wl.sps.cuda()
    lengths, B, theta = spec.spec_schedule_prefix(surv, sps, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    s = surv.cpu().numpy()
    assert np.all(np.diff(s, axis=1) <= 0) and np.all((s >= 0) & (s <= 1))
    sch = oracle.schedule_prefix(surv.cpu(), wl.sps.numpy())
    np.testing.assert_array_equal(lengths.cpu().numpy(), sch["lengths"])
    assert int(B.item()) == sch["B"] and float(theta.item()) == sch["theta"]
    sample = [0, 255, 256, 511]
    sl = lambda x: x[sample].cpu()
    ref = oracle.markov_propose(sl(wl.U), wl.W1.cpu(), wl.W2.cpu(), sl(wl.anchors),
                                sl(wl.u_draft), 1.0)
    compare_proposals(toks[sample], logp[sample], stats[sample], ref)
    tv = oracle.tv_confidence(sl(wl.U), sl(wl.target), wl.W1.cpu(), wl.W2.cpu(), sl(wl.anchors),
                              toks[sample].cpu(), 1.0)
    assert_conf_close(conf[sample], tv["conf"])
    assert_conf_close(surv[sample], tv["survival"], "survival")


def test_full_loop_full_size_sampled(spec):
    """R = 1024, gamma = 16, 20 chained iterations in one CUDA graph (Zipf prior, T = 0.7):
    every request's outputs are well formed, and a sample of requests is checked against the
    oracle at the first and the last iteration, given the GPU's state entering each."""
    from draft_sampling_verification_markov_gb300.loop import SpecLoop
    R, g, V, iters = 1024, 16, 129280, 20
    wl = W.full_loop("cuda", R=R, gamma=g, V=V, rank=256, iterations=iters, seed=1005)
    lp = SpecLoop(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, wl.u_draft, wl.u_accept,
                  wl.u_resid, wl.temperature, wl.sps.cuda())
    lp.capture()
    lp.replay()
    torch.cuda.synchronize()
    assert lp.ws.status() == 0
    n, o, ln = lp.accept_len.cpu().numpy(), lp.out_tokens.cpu().numpy(), lp.lengths.cpu().numpy()
    assert ((n >= 0) & (n <= ln)).all() and ((ln >= 0) & (ln <= g)).all()
    for t in range(iters):
        np.testing.assert_array_equal(lp.anchors[t + 1].cpu().numpy(), o[t, np.arange(R), n[t]])
    for t in (0, iters - 1):  # check_iteration copies the sampled rows to the host
        check_iteration(lp, wl, t, sample=[0, 511, 1023])
