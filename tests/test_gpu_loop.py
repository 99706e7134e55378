"""The device-resident draft -> verify loop (accepted prefix + emitted token; the emitted token
is the next iteration's anchor) against the oracle, iteration by iteration.

Each iteration is checked given the GPU's own state entering it (its anchors), so a sampled
token that legitimately differs at a CDF near-tie does not make the rest of the chain
incomparable: proposals, confidences, survival, scheduler lengths and verification outputs of
iteration t are compared with the oracle run on the GPU's anchors, draft tokens, survival and
lengths of iteration t."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import assert_conf_close, compare_proposals, compare_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def _loop(spec, wl, schedule=True, async_schedule=False, flat=False):
    from draft_sampling_verification_markov_gb300.loop import SpecLoop
    g = {k: v.cuda() for k, v in wl.tensors().items()}
    return SpecLoop(g["U"], g["target"], g["W1"], g["W2"], g["anchors"], g["u_draft"],
                    g["u_accept"], g["u_resid"], wl.temperature, g.get("sps"),
                    schedule=schedule, async_schedule=async_schedule, flat=flat)


def check_iteration(lp, wl, t, sample=None, report=None):
    """Teacher-forced oracle check of iteration t on the requests in `sample` (all by default)."""
    R = wl.R
    sample = list(range(R)) if sample is None else list(sample)
    sl = lambda x: x[sample].cpu()
    a_t = lp.anchors[t][sample].cpu()
    toks = lp.draft_tokens[t][sample].cpu()
    ref = oracle.markov_propose(sl(wl.U), wl.W1.cpu(), wl.W2.cpu(), a_t, sl(wl.u_draft[t]),
                                wl.temperature)
    # propose writes draft_logp / draft_stats only for the last iteration run; compare tokens
    # (margin rule) here and the probabilities through the confidence pass below
    compare_proposals(toks, None, None, ref, report=report)
    tv = oracle.tv_confidence(sl(wl.U), sl(wl.target), wl.W1.cpu(), wl.W2.cpu(), a_t, toks,
                              wl.temperature)
    if lp.schedule:
        assert_conf_close(lp.conf[t][sample], tv["conf"])
        assert_conf_close(lp.survival[t][sample], tv["survival"], "survival")
        # the scheduler sees every request: bit-exact on the GPU's survival
        sps = wl.sps.cpu().numpy()
        sch = oracle.schedule_prefix(lp.survival[t].cpu(), sps)
        if lp.async_schedule and t >= 2:
            # dynamic top-K: capacity = the Theta optimum of iteration t - 2's survival
            cap = oracle.schedule_prefix(lp.survival[t - 2].cpu(), sps)["B"]
            assert int(lp.batch_opt[t].item()) == sch["B"]
            sch = oracle.schedule_topk(lp.survival[t].cpu(), sps, cap)
        np.testing.assert_array_equal(lp.lengths[t].cpu().numpy(), sch["lengths"])
        assert int(lp.batch[t].item()) == sch["B"]
        assert float(lp.theta[t].item()) == sch["theta"]
        lengths = lp.lengths[t][sample].cpu()
    else:
        lengths = None
    rv = oracle.verify_rejection(sl(wl.target), sl(wl.U), wl.W1.cpu(), wl.W2.cpu(), a_t, toks,
                                 sl(wl.u_accept[t]), sl(wl.u_resid[t]), wl.temperature, lengths)
    n = lp.accept_len[t][sample].cpu().numpy()
    o = lp.out_tokens[t][sample].cpu().numpy()
    nxt = lp.anchors[t + 1][sample].cpu().numpy()
    # the oracle ran on the GPU's own draft tokens, so every request is compared
    compare_verify(n, o, nxt, rv, report=report)
    # the emitted token is the next anchor
    np.testing.assert_array_equal(nxt, o[np.arange(len(sample)), n])


@pytest.mark.parametrize("schedule", [True, False, "async"])
def test_loop_matches_oracle_iteration_by_iteration(spec, schedule):
    iters = 6 if schedule == "async" else 3
    wl = W.full_loop("cpu", R=6, gamma=4, V=1040, rank=64, iterations=iters, seed=31)
    lp = _loop(spec, wl, bool(schedule), async_schedule=schedule == "async")
    lp.run()
    torch.cuda.synchronize()
    assert lp.ws.status() == 0
    for t in range(wl.iterations):
        check_iteration(lp, wl, t)
    if not schedule:
        assert (lp.accept_len <= wl.gamma).all()


def test_loop_graph_replay_equals_eager(spec):
    wl = W.full_loop("cpu", R=70, gamma=5, V=2048, rank=128, iterations=4, seed=32)
    eager = _loop(spec, wl)
    eager.run()
    graph = _loop(spec, wl)
    graph.capture()
    graph.replay()
    torch.cuda.synchronize()
    for name in ("anchors", "draft_tokens", "conf", "survival", "lengths", "accept_len",
                 "out_tokens", "theta"):
        assert torch.equal(getattr(eager, name), getattr(graph, name)), name
    first = graph.out_tokens.clone()
    graph.replay()                       # replays start again from anchors[0]
    torch.cuda.synchronize()
    assert torch.equal(first, graph.out_tokens)
    assert eager.ws.status() == 0 and graph.ws.status() == 0


@pytest.mark.parametrize("async_schedule", [False, True])
def test_flat_loop_equals_padded_loop(spec, async_schedule):
    """Verification of the flattened batch (packed target rows and normalisers, per-request
    offsets) gives the padded loop's outputs bit for bit, eager and as one replayed graph."""
    wl = W.full_loop("cpu", R=70, gamma=5, V=2048, rank=128, iterations=4, seed=36)
    padded = _loop(spec, wl, async_schedule=async_schedule)
    padded.run()
    flat = _loop(spec, wl, async_schedule=async_schedule, flat=True)
    flat.run()
    graph = _loop(spec, wl, async_schedule=async_schedule, flat=True)
    graph.capture()
    graph.replay()
    torch.cuda.synchronize()
    for name in ("anchors", "draft_tokens", "lengths", "batch", "accept_len", "out_tokens"):
        assert torch.equal(getattr(padded, name), getattr(flat, name)), name
        assert torch.equal(getattr(padded, name), getattr(graph, name)), name
    # the packed rows of the last iteration are the scheduled rows, in request order
    B = int(flat.batch[-1])
    assert int(flat.offsets[-1]) == B
    ln = flat.lengths[-1].cpu()
    rows = [r * (wl.gamma + 1) + i for r in range(wl.R) for i in range(int(ln[r]) + 1)]
    want = flat.target.view(-1, wl.V)[torch.tensor(rows, device="cuda")]
    assert torch.equal(flat.packed_target[:B], want)
    assert padded.ws.status() == 0 and flat.ws.status() == 0 and graph.ws.status() == 0


def test_async_loop_graph_replay_equals_eager(spec):
    """The asynchronous scheduler's capacity history lives on the device, so a captured graph of
    the whole loop reproduces the eager run, including the top-K lengths."""
    wl = W.full_loop("cpu", R=40, gamma=5, V=2048, rank=64, iterations=6, seed=35)
    eager = _loop(spec, wl, async_schedule=True)
    eager.run()
    graph = _loop(spec, wl, async_schedule=True)
    graph.capture()
    graph.replay()
    torch.cuda.synchronize()
    for name in ("anchors", "lengths", "batch", "accept_len", "out_tokens", "theta"):
        assert torch.equal(getattr(eager, name), getattr(graph, name)), name
    assert torch.equal(eager.batch_opt[2:], graph.batch_opt[2:])
    assert eager.ws.status() == 0 and graph.ws.status() == 0


def test_loop_resumes_from_an_iteration(spec):
    """Stopping after iteration 1 and resuming at iteration 2 (from the stored anchors) gives the
    same outputs as one uninterrupted run."""
    wl = W.full_loop("cpu", R=9, gamma=3, V=1040, rank=64, iterations=4, seed=33)
    whole = _loop(spec, wl)
    whole.run()
    split = _loop(spec, wl)
    split.run(0, 2)
    torch.cuda.synchronize()
    resumed = _loop(spec, wl)
    resumed.anchors[2].copy_(split.anchors[2])          # the saved loop state
    resumed.run(2, 4)
    torch.cuda.synchronize()
    for name in ("draft_tokens", "accept_len", "out_tokens", "lengths"):
        a, b, c = getattr(whole, name), getattr(split, name), getattr(resumed, name)
        assert torch.equal(a[:2], b[:2]), name
        assert torch.equal(a[2:], c[2:]), name
    assert torch.equal(whole.anchors[4], resumed.anchors[4])
