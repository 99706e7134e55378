"""Sparse target distributions (vocab-shuffled Zipf prior; top-k / top-p truncated target rows,
-inf outside the nucleus) through the CUDA path against the oracle: proposals, target
normalisers, rejection verification with residual / bonus draws, TV confidence, and greedy
verification. Properties that hold for any truncation are checked on every request: an
accepted draft token lies in its target row's nucleus, and so does every final draw."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import assert_conf_close, compare_proposals, compare_verify, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


CASES = [dict(top_k=20), dict(top_p=0.9), dict(top_k=None)]


def _check_nucleus(target, tokens, n, out, gamma):
    fin = torch.isfinite(target.float()).cpu().numpy()           # [R, gamma+1, V]
    t, nn, o = tokens.cpu().numpy(), n.cpu().numpy(), out.cpu().numpy()
    for r in range(t.shape[0]):
        for k in range(nn[r]):                                  # accepted x_{k+1} vs row k
            assert fin[r, k, t[r, k]], (r, k)
        assert fin[r, nn[r], o[r, nn[r]]], r                    # the final draw, row n


@pytest.mark.parametrize("case", CASES, ids=["top_k20", "top_p0.9", "zipf_only"])
@pytest.mark.parametrize("T", [1.0, 0.8])
def test_sparse_targets_match_oracle(spec, case, T):
    wl = W.sparse_targets("cpu", R=70, gamma=4, V=2048, rank=64, seed=61, temperature=T, **case)
    g = to_dev(wl, "cuda")
    ws = spec.Workspace(device="cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"],
                                                 g["u_draft"], T, workspace=ws)
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, T)
    same = compare_proposals(toks, logp, stats, ref)
    tst = spec.spec_target_stats(g["target"], T, workspace=ws)
    n, out, nxt = spec.spec_verify_rejection(g["target"], g["U"], g["W1"], g["W2"], g["anchors"],
                                             toks, logp, stats, g["u_accept"], g["u_resid"], T,
                                             target_stats=tst, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _check_nucleus(wl.target, toks, n, out, wl.gamma)
    rv = oracle.verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, toks.cpu(),
                                 wl.u_accept, wl.u_resid, T)
    compare_verify(n.cpu().numpy(), out.cpu().numpy(), None, rv)
    # TV confidence on the GPU's proposals
    conf, surv = spec.spec_tv_confidence(g["U"], g["target"], g["W1"], g["W2"], g["anchors"],
                                         toks, T, draft_stats=stats, target_stats=tst,
                                         workspace=ws)
    tv = oracle.tv_confidence(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, toks.cpu(), T)
    assert_conf_close(conf, tv["conf"])
    assert_conf_close(surv, tv["survival"], "survival")
    # greedy verify of the same proposals: bit-exact
    gn2, go2, gx2 = spec.spec_verify_greedy(g["target"], toks, workspace=ws)
    rg = oracle.verify_greedy(wl.target, toks.cpu())
    np.testing.assert_array_equal(gn2.cpu().numpy(), rg["accept_len"])
    np.testing.assert_array_equal(go2.cpu().numpy(), rg["out_tokens"])


def test_top_k_full_size_sampled(spec):
    """The benchmarked shapes (R = 256, gamma = 7, V = 129280, rank 256) with top-50 targets:
    nucleus properties on every request, oracle on a sample."""
    R, g_, V = 256, 7, 129280
    wl = W.sparse_targets("cuda", R=R, gamma=g_, V=V, rank=256, top_k=50)
    ws = spec.Workspace(device="cuda")
    toks, logp, stats = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, 1.0,
                                                 workspace=ws)
    n, out, nxt = spec.spec_verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, toks,
                                             logp, stats, wl.u_accept, wl.u_resid, 1.0,
                                             workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    _check_nucleus(wl.target, toks, n, out, g_)
    sample = [0, 127, 128, 255]
    sl = lambda x: x[sample].cpu()
    rv = oracle.verify_rejection(sl(wl.target), sl(wl.U), wl.W1.cpu(), wl.W2.cpu(),
                                 sl(wl.anchors), toks[sample].cpu(), sl(wl.u_accept),
                                 sl(wl.u_resid), 1.0)
    amb = (np.nan_to_num(rv["accept_margin"], nan=1.0) < 1e-6).any(axis=1) | (
        rv["resid_margin"] < 1e-6)
    for si, r in enumerate(sample):
        if not amb[si]:
            assert n[r].item() == rv["accept_len"][si]
            np.testing.assert_array_equal(out[r].cpu().numpy(), rv["out_tokens"][si])
