"""Parity at the full sizes of the workloads, in the launch configuration bench.py times: the
whole batch runs on the GPU and the oracle recomputes every request (requests are independent in
proposal and verification), except in the 20-iteration loop, where 64 requests spread over all
row blocks are recomputed at the first, a middle and the last iteration. Properties that hold at
any size are checked on every request, and the share of requests identical to the oracle is
asserted (a mismatch is only allowed at a CDF or acceptance margin below 1e-6, which the
synthetic inputs almost never produce)."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import LOG_TOL, assert_conf_close, compare_proposals, compare_verify
from test_gpu_loop import check_iteration

pytestmark = pytest.mark.gpu

# the least share of requests whose outputs must equal the oracle's exactly
MIN_EXACT = 0.99


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def _norm_errors(stats, target, T):
    """|(m + log Z) - fp64 log-sum-exp| / max(1, |.|) for every row of target / T."""
    inv = float(np.float32(1) / np.float32(T))
    st = stats.cpu().numpy().astype(np.float64)
    errs = []
    for chunk in torch.split(target.reshape(-1, target.shape[-1]), 256):
        z = chunk.double().cpu().numpy() * inv
        m = z.max(axis=1)
        errs.append(m + np.log(np.exp(z - m[:, None]).sum(axis=1)))
    want = np.concatenate(errs)
    return np.abs((st[:, 0] + st[:, 1]) - want) / np.maximum(1.0, np.abs(want))


@pytest.mark.parametrize("fused", [False, True])
def test_markov_rejection_full_size_all_requests(spec, fused):
    """R = 256, gamma = 7, V = 129280 (the benchmarked workload): every request's proposals,
    target normalisers and verification against the oracle."""
    R, g, V = 256, 7, 129280
    wl = W.markov_rejection("cuda", R=R, gamma=g, V=V, rank=256, seed=1003)
    ws = spec.Workspace(device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())  # the inputs are drawn on the current stream
    with torch.cuda.stream(stream):
        if fused:
            toks, logp, stats, tst = spec.spec_markov_propose_target_stats(
                wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, 1.0, wl.target, workspace=ws,
                stream=stream)
        else:
            toks, logp, stats = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors,
                                                         wl.u_draft, 1.0, workspace=ws,
                                                         stream=stream)
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
    # the oracle on every request
    c = lambda x: x.cpu()
    ref = oracle.markov_propose(c(wl.U), c(wl.W1), c(wl.W2), c(wl.anchors), c(wl.u_draft), 1.0)
    same = compare_proposals(toks, logp, stats, ref)
    assert same.mean() >= MIN_EXACT, f"only {same.sum()} of {R} proposals identical"
    rv = oracle.verify_rejection(c(wl.target), c(wl.U), c(wl.W1), c(wl.W2), c(wl.anchors),
                                 ref["tokens"], c(wl.u_accept), c(wl.u_resid), 1.0)
    compared = compare_verify(nn, o, nxt.cpu().numpy(), rv, same)
    assert compared >= MIN_EXACT * R
    # target normalisers of every row
    assert _norm_errors(tst, wl.target, 1.0).max() <= LOG_TOL


def test_confidence_scheduling_full_size_all_requests(spec):
    """R = 512, gamma = 16: proposal, target normalisers, TV confidence with survival on every
    request, and the scheduler over all 8192 candidates (bit-exact on the GPU's survival)."""
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
    c = lambda x: x.cpu()
    ref = oracle.markov_propose(c(wl.U), c(wl.W1), c(wl.W2), c(wl.anchors), c(wl.u_draft), 1.0)
    same = compare_proposals(toks, logp, stats, ref)
    assert same.mean() >= MIN_EXACT, f"only {same.sum()} of {R} proposals identical"
    # the labels of the GPU's own proposals (defined for any proposal)
    tv = oracle.tv_confidence(c(wl.U), c(wl.target), c(wl.W1), c(wl.W2), c(wl.anchors),
                              toks.cpu(), 1.0)
    assert_conf_close(conf, tv["conf"])
    assert_conf_close(surv, tv["survival"], "survival")


def test_full_loop_full_size_sampled(spec):
    """R = 1024, gamma = 16, 20 chained iterations in one CUDA graph (Zipf prior, T = 0.7):
    every request's outputs are well formed, and 64 requests spread over all row blocks are
    checked against the oracle at the first, a middle and the last iteration, given the GPU's
    state entering each."""
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
    sample = np.linspace(0, R - 1, 64).round().astype(int).tolist()
    for t in (0, iters // 2 - 1, iters - 1):  # check_iteration copies the sampled rows to the host
        check_iteration(lp, wl, t, sample=sample)
