"""Degenerate shapes through the C ABI against the oracle: no requests, no draft positions (the
verify window is the bonus row alone), and a one-token vocabulary (every distribution is a point
mass, so every proposal is accepted and every confidence is 1)."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


@pytest.fixture()
def ws(spec):
    w = spec.Workspace(device="cuda")
    yield w
    torch.cuda.synchronize()
    assert w.status() == 0, "device status word set"


def test_no_requests(spec, ws):
    V, gamma, rank = 1000, 3, 64
    e = dict(device="cuda")
    U = torch.empty(0, gamma, V, dtype=torch.bfloat16, **e)
    T = torch.empty(0, gamma + 1, V, dtype=torch.bfloat16, **e)
    W1 = torch.zeros(V, rank, dtype=torch.bfloat16, **e)
    W2 = torch.zeros(V, rank, dtype=torch.bfloat16, **e)
    anchors = torch.empty(0, dtype=torch.int32, **e)
    u = torch.empty(0, gamma, **e)
    toks, logp, st = spec.spec_markov_propose(U, W1, W2, anchors, u, 1.0, workspace=ws)
    assert toks.shape == (0, gamma)
    n, out, nxt = spec.spec_verify_greedy(T, toks, workspace=ws)
    assert n.numel() == 0 and out.shape == (0, gamma + 1)
    n, out, nxt = spec.spec_verify_rejection(T, U, W1, W2, anchors, toks, logp, st, u,
                                             torch.empty(0, **e), 1.0, workspace=ws)
    assert n.numel() == 0
    conf, surv = spec.spec_tv_confidence(U, T, W1, W2, anchors, toks, 1.0, workspace=ws)
    assert conf.shape == (0, gamma)
    lengths, B, theta = spec.spec_schedule_prefix(torch.empty(0, gamma, **e),
                                                  torch.ones(5, dtype=torch.float64, **e),
                                                  workspace=ws)
    assert int(B.item()) == 0


@pytest.mark.parametrize("rank", [0, 64])
def test_no_draft_positions(spec, ws, rank):
    """gamma = 0: greedy verify emits the target argmax of row 0, rejection verify draws from
    p_t of row 0 with the residual uniform."""
    R, V = 37, 4104
    wl = W.markov_rejection("cpu", R=R, gamma=1, V=V, rank=64, seed=91, temperature=0.9)
    T0 = wl.target[:, :1].contiguous()
    U0 = wl.U[:, :0].contiguous()
    W1 = wl.W1 if rank else None
    W2 = wl.W2 if rank else None
    d = lambda x: None if x is None else x.cuda()
    toks = torch.empty(R, 0, dtype=torch.int32, device="cuda")
    n, out, nxt = spec.spec_verify_greedy(T0.cuda(), toks, workspace=ws)
    rg = oracle.verify_greedy(T0, toks.cpu())
    np.testing.assert_array_equal(n.cpu().numpy(), rg["accept_len"])
    np.testing.assert_array_equal(nxt.cpu().numpy(), rg["next_anchor"])
    e = torch.empty(R, 0, device="cuda")
    n, out, nxt = spec.spec_verify_rejection(
        T0.cuda(), U0.cuda(), d(W1), d(W2), wl.anchors.cuda(), toks, e, torch.empty(R, 0, 2, device="cuda"),
        e, wl.u_resid.cuda(), 0.9, rank=rank, workspace=ws)
    rv = oracle.verify_rejection(T0, U0, W1, W2, wl.anchors, toks.cpu(), wl.u_accept[:, :0],
                                 wl.u_resid, 0.9, rank=rank)
    assert (n.cpu().numpy() == 0).all()
    gx = nxt.cpu().numpy()
    diff = gx != rv["next_anchor"]
    assert not (diff & ~(rv["resid_margin"] < 1e-6)).any()


def test_one_token_vocabulary(spec, ws):
    """V = 1: the proposal is token 0 everywhere, every position is accepted (p_d = p_t = 1),
    the bonus is token 0, and every confidence and survival is exactly 1."""
    R, gamma, V, rank = 9, 4, 1, 16
    g = torch.Generator().manual_seed(5)
    U = torch.randn(R, gamma, V, generator=g).cuda()
    T = torch.randn(R, gamma + 1, V, generator=g).cuda()
    W1 = torch.randn(V, rank, generator=g).cuda()
    W2 = torch.randn(V, rank, generator=g).cuda()
    anchors = torch.zeros(R, dtype=torch.int32, device="cuda")
    u = torch.rand(R, gamma, generator=g).cuda()
    toks, logp, st = spec.spec_markov_propose(U, W1, W2, anchors, u, 1.0, workspace=ws)
    assert (toks == 0).all() and (logp == 0).all()
    n, out, nxt = spec.spec_verify_rejection(T, U, W1, W2, anchors, toks, logp, st, u,
                                             torch.rand(R, generator=g).cuda(), 1.0,
                                             workspace=ws)
    assert (n == gamma).all() and (nxt == 0).all() and (out == 0).all()
    conf, surv = spec.spec_tv_confidence(U, T, W1, W2, anchors, toks, 1.0, draft_stats=st,
                                         workspace=ws)
    assert (conf == 1).all() and (surv == 1).all()
    n, out, nxt = spec.spec_verify_greedy(T, toks, workspace=ws)
    assert (n == gamma).all() and (nxt == 0).all()


@pytest.mark.parametrize("R,V", [(200, 4104), (600, 129280)])
def test_w1_alignment_16_bytes(spec, ws, R, V):
    """The tensor-core pass reads W1 rows with 32-byte loads when W1 is 32-byte aligned and
    with 16-byte loads otherwise: a W1 at a 16-byte offset gives bit-identical proposals and
    residual draws. At R = 600 the CTAs' unit ranges cross row-block pairs, so the gather of a
    CTA's later pair (16-byte loads either way) runs too."""
    gamma, rank = 4, 256
    wl = W.markov_rejection("cuda", R=R, gamma=gamma, V=V, rank=rank, seed=77, temperature=1.0)
    buf = torch.empty(V * rank + 8, dtype=wl.W1.dtype, device="cuda")
    W1_off = buf[8:].view(V, rank)
    W1_off.copy_(wl.W1)
    assert W1_off.data_ptr() % 32 == 16
    outs = []
    for W1 in (wl.W1, W1_off):
        toks, logp, st = spec.spec_markov_propose(wl.U, W1, wl.W2, wl.anchors, wl.u_draft, 1.0,
                                                  workspace=ws)
        n, out, nxt = spec.spec_verify_rejection(wl.target, wl.U, W1, wl.W2, wl.anchors, toks,
                                                 logp, st, wl.u_accept, wl.u_resid, 1.0,
                                                 workspace=ws)
        outs.append([x.cpu() for x in (toks, logp, st, n, out, nxt)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
