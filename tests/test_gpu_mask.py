"""Grammar-masked drafting through the CUDA path against the oracle: the draft distribution of a
masked request is restricted to its allowed tokens (bitmask [R, ceil(V/32)]), in the proposal
(tensor-core, CUDA-core and rank-0 streaming producers), in the rejection residual and in the TV
label. Every proposed token must be allowed; an all-ones mask must give the unmasked results."""
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


def _mask(R, V, frac, seed, always=(0,)):
    rng = np.random.default_rng(seed)
    allowed = rng.random((R, V)) < frac
    allowed[:, list(always)] = True
    words = np.zeros((R, (V + 31) // 32), dtype=np.uint32)
    for r in range(R):
        idx = np.nonzero(allowed[r])[0]
        np.bitwise_or.at(words[r], idx // 32, (np.uint32(1) << (idx % 32).astype(np.uint32)))
    return allowed, torch.from_numpy(words.view(np.int32))


def _wl(R, gamma, V, rank, wdt, seed, T):
    wl = W.markov_rejection("cpu", R=R, gamma=gamma, V=V, rank=max(rank, 1), seed=seed,
                            temperature=T)
    if rank == 0:
        wl.W1 = wl.W2 = None
        wl.rank = 0
    elif wdt == "f32":
        wl.W1, wl.W2 = wl.W1.float(), wl.W2.float()
        wl.U, wl.target = wl.U.float(), wl.target.float()
    return wl


# tensor-core (bf16, rank % 64 == 0, V % 8 == 0), CUDA-core (fp32 / odd rank) and streaming
CASES = [(70, 4, 2048, 64, "bf16"), (70, 3, 1000, 40, "f32"), (33, 3, 3000, 0, "bf16")]


@pytest.mark.parametrize("R,gamma,V,rank,wdt", CASES)
def test_masked_sampling_propose_verify_and_confidence(spec, R, gamma, V, rank, wdt):
    T = 0.9
    wl = _wl(R, gamma, V, rank, wdt, seed=70 + V, T=T)
    allowed, words = _mask(R, V, 0.1, seed=V)
    mask_np = words.numpy().view(np.uint32)
    g = to_dev(wl, "cuda")
    m = words.cuda()
    ws = spec.Workspace(device="cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g.get("W1"), g.get("W2"), g["anchors"],
                                                 g["u_draft"], T, rank=rank, workspace=ws,
                                                 allowed=m)
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, T, rank=rank,
                                mask=mask_np)
    compare_proposals(toks, logp, stats, ref)
    t = toks.cpu().numpy()
    assert all(allowed[r, t[r, k]] for r in range(R) for k in range(gamma))
    n, out, nxt = spec.spec_verify_rejection(g["target"], g["U"], g.get("W1"), g.get("W2"),
                                             g["anchors"], toks, logp, stats, g["u_accept"],
                                             g["u_resid"], T, rank=rank, workspace=ws, allowed=m)
    rv = oracle.verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, toks.cpu(),
                                 wl.u_accept, wl.u_resid, T, rank=rank, mask=mask_np)
    compare_verify(n.cpu().numpy(), out.cpu().numpy(), None, rv)
    conf, surv = spec.spec_tv_confidence(g["U"], g["target"], g.get("W1"), g.get("W2"),
                                         g["anchors"], toks, T, rank=rank, draft_stats=stats,
                                         workspace=ws, allowed=m)
    tv = oracle.tv_confidence(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, toks.cpu(), T,
                              rank=rank, mask=mask_np)
    assert_conf_close(conf, tv["conf"])
    assert_conf_close(surv, tv["survival"], "survival")
    torch.cuda.synchronize()
    assert ws.status() == 0


def test_masked_greedy_is_bit_exact_on_the_fp32_path(spec):
    wl = W.greedy_toy("cpu", R=5, gamma=4, V=1000, rank=40, seed=71)
    allowed, words = _mask(5, 1000, 0.05, seed=3)
    g = to_dev(wl, "cuda")
    ws = spec.Workspace(device="cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"], None, 0.0,
                                                 workspace=ws, allowed=words.cuda())
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, None, 0.0,
                                mask=words.numpy().view(np.uint32))
    compare_proposals(toks, logp, stats, ref, greedy=True)


def test_masked_mtp_argmax(spec):
    """rank 0 (MTP/NextN) greedy argmax restricted to the allowed tokens, at the full
    vocabulary: bit-exact token ids."""
    wl = W.mtp_greedy("cpu", R=9, gamma=3, V=129280, seed=72)
    allowed, words = _mask(9, 129280, 0.01, seed=4)
    g = to_dev(wl, "cuda")
    ws = spec.Workspace(device="cuda")
    toks, _, _ = spec.spec_markov_propose(g["U"], None, None, None, None, 0.0, workspace=ws,
                                          allowed=words.cuda())
    ref = oracle.markov_propose(wl.U, None, None, None, None, 0.0,
                                mask=words.numpy().view(np.uint32))
    np.testing.assert_array_equal(toks.cpu().numpy(), ref["tokens"])
    u = wl.U.float().numpy()
    for r in range(9):
        for k in range(3):
            assert toks[r, k].item() == int(np.argmax(np.where(allowed[r], u[r, k], -np.inf)))


def test_all_ones_mask_equals_no_mask(spec):
    wl = W.markov_rejection("cuda", R=130, gamma=3, V=4096, rank=128, seed=73)
    ones = torch.full((130, 128), -1, dtype=torch.int32, device="cuda")
    ws = spec.Workspace(device="cuda")
    a = [x.clone() for x in spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft,
                                                     1.0, workspace=ws)]
    b = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, 1.0, workspace=ws,
                                 allowed=ones)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_masked_loop_iterations_match_oracle(spec):
    """The device-resident loop with a grammar mask: every iteration's proposals, confidences,
    scheduler lengths and verification against the oracle given the GPU's anchors, and every
    drafted token allowed."""
    from draft_sampling_verification_markov_gb300.loop import SpecLoop
    R, gamma, V = 6, 4, 1040
    wl = W.full_loop("cpu", R=R, gamma=gamma, V=V, rank=64, iterations=3, seed=41)
    allowed, words = _mask(R, V, 0.3, 9)
    g = {k: v.cuda() for k, v in wl.tensors().items()}
    lp = SpecLoop(g["U"], g["target"], g["W1"], g["W2"], g["anchors"], g["u_draft"],
                  g["u_accept"], g["u_resid"], wl.temperature, g["sps"], allowed=words.cuda())
    lp.run()
    torch.cuda.synchronize()
    assert lp.ws.status() == 0
    mask = words.numpy()
    for t in range(wl.iterations):
        a_t = lp.anchors[t].cpu()
        toks = lp.draft_tokens[t].cpu()
        tk = toks.numpy()
        assert allowed[np.arange(R)[:, None], tk].all()
        ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, a_t, wl.u_draft[t], wl.temperature,
                                    mask=mask)
        compare_proposals(toks, None, None, ref)
        tv = oracle.tv_confidence(wl.U, wl.target, wl.W1, wl.W2, a_t, toks, wl.temperature,
                                  mask=mask)
        assert_conf_close(lp.conf[t], tv["conf"])
        sch = oracle.schedule_prefix(lp.survival[t].cpu(), wl.sps.numpy())
        np.testing.assert_array_equal(lp.lengths[t].cpu().numpy(), sch["lengths"])
        rv = oracle.verify_rejection(wl.target, wl.U, wl.W1, wl.W2, a_t, toks, wl.u_accept[t],
                                     wl.u_resid[t], wl.temperature, lp.lengths[t].cpu(),
                                     mask=mask)
        n = lp.accept_len[t].cpu().numpy()
        nxt = lp.anchors[t + 1].cpu().numpy()
        o = lp.out_tokens[t].cpu().numpy()
        compare_verify(n, o, nxt, rv)
