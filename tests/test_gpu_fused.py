"""The fused proposal + target normalisers entry point (spec_markov_propose_target_stats)
against the oracle: the proposals follow the same comparison rules as spec_markov_propose, the
target normalisers are checked against a float64 log-sum-exp of every row, and rejection
verification with those normalisers against the oracle's. Shapes cover the persistent
tensor-core launch (one and two request groups, a ragged last group), the persistent proposal
followed by a separate normaliser pass (more than two groups), and the fallback of two separate
passes (fp32 weights, no Markov head, no draft positions)."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import LOG_TOL, compare_proposals, compare_verify, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def _target_norms(target, T):
    """(m + log Z) of softmax(target / T) per row, float64 (the scale is fl32(1 / T))."""
    z = target.double().reshape(-1, target.shape[-1]).numpy() * float(np.float32(1) / np.float32(T))
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


@pytest.mark.parametrize("R,gamma,V,rank,wdt", [
    (300, 2, 4104, 128, "bf16"),   # persistent proposal, three groups: normalisers after it
    (130, 3, 4104, 128, "bf16"),   # persistent: two groups, the second of two rows
    (9, 4, 2048, 256, "bf16"),     # persistent: one group
    (7, 3, 1000, 48, "f32"),       # two passes: fp32 weights on CUDA cores
    (5, 2, 2048, 0, "bf16"),       # two passes: no Markov head
])
def test_fused_propose_and_target_stats(spec, R, gamma, V, rank, wdt):
    T = 0.8
    wl = W.markov_rejection("cpu", R=R, gamma=gamma, V=V, rank=max(rank, 1), seed=300 + V,
                            temperature=T)
    if rank == 0:
        wl.W1 = wl.W2 = None
    elif wdt == "f32":
        wl.W1, wl.W2 = wl.W1.float(), wl.W2.float()
        wl.U, wl.target = wl.U.float(), wl.target.float()
    g = to_dev(wl, "cuda")
    ws = spec.Workspace(device="cuda")
    toks, logp, stats, tst = spec.spec_markov_propose_target_stats(
        g["U"], g.get("W1"), g.get("W2"), g["anchors"], g["u_draft"], T, g["target"], rank=rank,
        workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, T, rank=rank)
    same = compare_proposals(toks, logp, stats, ref)
    assert same.mean() > 0.9
    st = tst.cpu().numpy().astype(np.float64)
    want = _target_norms(wl.target, T)
    err = np.abs((st[:, 0] + st[:, 1]) - want) / np.maximum(1.0, np.abs(want))
    assert err.max() <= LOG_TOL, f"target normaliser differs by {err.max():.3e}"
    n, out, nxt = spec.spec_verify_rejection(g["target"], g["U"], g.get("W1"), g.get("W2"),
                                             g["anchors"], toks, logp, stats, g["u_accept"],
                                             g["u_resid"], T, rank=rank, target_stats=tst,
                                             workspace=ws)
    rv = oracle.verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, ref["tokens"],
                                 wl.u_accept, wl.u_resid, T, rank=rank)
    compare_verify(n.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy(), rv, same)
    assert ws.status() == 0


def test_fused_without_draft_positions(spec):
    """gamma = 0: nothing is proposed; the bonus rows' normalisers are still written."""
    wl = W.markov_rejection("cpu", R=3, gamma=1, V=512, rank=64, seed=5)
    target = wl.target[:, :1].contiguous().cuda()
    U = torch.empty(3, 0, 512, dtype=torch.bfloat16, device="cuda")
    toks, logp, stats, tst = spec.spec_markov_propose_target_stats(
        U, wl.W1.cuda(), wl.W2.cuda(), wl.anchors.cuda(), None, 1.0, target)
    torch.cuda.synchronize()
    want = _target_norms(target.cpu(), 1.0)
    st = tst.cpu().numpy().astype(np.float64)
    assert np.abs((st[:, 0] + st[:, 1]) - want).max() <= LOG_TOL * max(1.0, np.abs(want).max())


def test_fused_rejects_missing_target(spec):
    wl = W.markov_rejection("cpu", R=2, gamma=2, V=512, rank=64, seed=5)
    g = to_dev(wl, "cuda")
    ws = spec.Workspace(device="cuda")
    wp, wn = ws.for_op(spec.SPEC_OP_PROPOSE, 2, 2, 512, 64)
    toks = torch.empty(2, 2, dtype=torch.int32, device="cuda")
    rc = spec.lib().spec_markov_propose_target_stats(
        spec._ptr(g["U"]), spec.SPEC_BF16, spec._ptr(g["W1"]), spec._ptr(g["W2"]), spec.SPEC_BF16,
        64, spec._ptr(g["anchors"]), spec._ptr(g["u_draft"]), 1.0, 2, 2, 512, spec._ptr(toks),
        None, None, None, None, wp, wn, None)
    assert rc == -1  # SPEC_ERR_INVALID_ARG
