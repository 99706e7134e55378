"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded bytes.

Sizes here span several tiles and a ragged tail and finish in seconds on the oracle; the
full-size workloads are covered in test_gpu_fullsize.py."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import (assert_conf_close, compare_proposals, compare_verify, to_dev, LOG_TOL)

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


# ----------------------------------------------------------------------------- greedy paths

@pytest.mark.parametrize("R,gamma,V,rank", [(4, 4, 1000, 256), (3, 2, 8, 16), (5, 3, 777, 33)])
def test_greedy_f32_markov_bit_exact(spec, ws, R, gamma, V, rank):
    wl = W.greedy_toy("cpu", R=R, gamma=gamma, V=V, rank=rank, seed=11 + V)
    g = to_dev(wl, "cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"], None, 0.0,
                                                 workspace=ws)
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, None, 0.0)
    compare_proposals(toks, logp, stats, ref, greedy=True)
    n, out, nxt = spec.spec_verify_greedy(g["target"], toks, workspace=ws)
    rv = oracle.verify_greedy(wl.target, ref["tokens"])
    np.testing.assert_array_equal(n.cpu().numpy(), rv["accept_len"])
    np.testing.assert_array_equal(out.cpu().numpy(), rv["out_tokens"])
    np.testing.assert_array_equal(nxt.cpu().numpy(), rv["next_anchor"])


def test_greedy_toy_at_its_size_bit_exact(spec, ws):
    """The greedy toy workload at its own size (R = 4, gamma = 4, V = 32000, rank 256, fp32
    weights, inputs drawn as the bench draws them): greedy proposals on the canonical fp32 chain,
    greedy verification, accept lengths and bonus tokens bit for bit."""
    wl = W.greedy_toy("cuda", R=4, gamma=4, V=32000, rank=256, seed=1001)
    toks, logp, stats = spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, None, 0.0,
                                                 workspace=ws)
    c = lambda x: x.cpu()
    ref = oracle.markov_propose(c(wl.U), c(wl.W1), c(wl.W2), c(wl.anchors), None, 0.0)
    compare_proposals(toks, logp, stats, ref, greedy=True)
    n, out, nxt = spec.spec_verify_greedy(wl.target, toks, workspace=ws)
    rv = oracle.verify_greedy(c(wl.target), ref["tokens"])
    np.testing.assert_array_equal(n.cpu().numpy(), rv["accept_len"])
    np.testing.assert_array_equal(out.cpu().numpy(), rv["out_tokens"])
    np.testing.assert_array_equal(nxt.cpu().numpy(), rv["next_anchor"])


def test_mtp_greedy_at_its_size_bit_exact(spec, ws):
    """MTP-1 greedy verification at its own size (R = 64, gamma = 3, V = 129280, bf16, inputs
    drawn as the bench draws them): argmax proposals, the planted tokens, accept lengths and
    bonus tokens bit for bit."""
    wl = W.mtp_greedy("cuda", R=64, gamma=3, V=129280, seed=1002)
    toks, logp, stats = spec.spec_markov_propose(wl.U, None, None, None, None, 0.0,
                                                 workspace=ws)
    ref = oracle.markov_propose(wl.U.cpu(), None, None, None, None, 0.0)
    compare_proposals(toks, logp, stats, ref, greedy=True)
    np.testing.assert_array_equal(toks.cpu().numpy(), wl.extra["planted_tokens"].cpu().numpy())
    n, out, nxt = spec.spec_verify_greedy(wl.target, toks, workspace=ws)
    rv = oracle.verify_greedy(wl.target.cpu(), ref["tokens"])
    np.testing.assert_array_equal(n.cpu().numpy(), rv["accept_len"])
    np.testing.assert_array_equal(out.cpu().numpy(), rv["out_tokens"])
    np.testing.assert_array_equal(nxt.cpu().numpy(), rv["next_anchor"])


@pytest.mark.parametrize("V", [129280, 1003, 64])
def test_mtp_argmax_and_greedy_verify_bit_exact(spec, ws, V):
    wl = W.mtp_greedy("cpu", R=17, gamma=3, V=V, seed=5)
    g = to_dev(wl, "cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], None, None, None, None, 0.0,
                                                 workspace=ws)
    ref = oracle.markov_propose(wl.U, None, None, None, None, 0.0)
    compare_proposals(toks, logp, stats, ref, greedy=True)
    np.testing.assert_array_equal(toks.cpu().numpy(), wl.extra["planted_tokens"].numpy())
    for lengths in (None, torch.tensor([i % 4 for i in range(17)], dtype=torch.int32)):
        n, out, nxt = spec.spec_verify_greedy(
            g["target"], toks, None if lengths is None else lengths.cuda(), workspace=ws)
        rv = oracle.verify_greedy(wl.target, ref["tokens"], lengths)
        np.testing.assert_array_equal(n.cpu().numpy(), rv["accept_len"])
        np.testing.assert_array_equal(out.cpu().numpy(), rv["out_tokens"])
        np.testing.assert_array_equal(nxt.cpu().numpy(), rv["next_anchor"])


def test_greedy_ties_go_to_lowest_index(spec, ws):
    V = 300
    U = torch.zeros(2, 1, V, dtype=torch.bfloat16)
    U[0, 0, [17, 200, 299]] = 5.0
    U[1, 0, :] = 1.0                                   # all equal -> token 0
    toks, _, _ = spec.spec_markov_propose(U.cuda(), None, None, None, None, 0.0, workspace=ws)
    assert toks.cpu().tolist() == [[17], [0]]
    T = torch.zeros(1, 2, V, dtype=torch.bfloat16)
    T[0, 0, [5, 9]] = 3.0
    T[0, 1, 250:] = 2.0
    n, out, nxt = spec.spec_verify_greedy(T.cuda(), torch.tensor([[5]], dtype=torch.int32).cuda(),
                                          workspace=ws)
    assert n.item() == 1 and out.cpu().tolist() == [[5, 250]] and nxt.item() == 250


# ----------------------------------------------------------------------------- sampling paths

SAMPLING_CASES = [
    # R, gamma, V, rank, wdtype
    (130, 3, 1000, 256, "bf16"),     # two 128-row tiles, ragged vocab tail
    (9, 4, 4104, 64, "bf16"),
    (6, 3, 777, 32, "bf16"),         # V % 8 != 0 and rank % 64 != 0 (CUDA-core producer)
    (7, 3, 1000, 48, "f32"),         # fp32 weights: canonical fp32 chain
    (5, 4, 2048, 0, "bf16"),         # no Markov head
]


def _wl(R, gamma, V, rank, wdt, seed, T=1.0):
    wl = W.markov_rejection("cpu", R=R, gamma=gamma, V=V, rank=max(rank, 1), seed=seed,
                            temperature=T)
    if rank == 0:
        wl.W1 = wl.W2 = None
        wl.rank = 0
    elif wdt == "f32":
        wl.W1, wl.W2 = wl.W1.float(), wl.W2.float()
        wl.U, wl.target = wl.U.float(), wl.target.float()
    return wl


@pytest.mark.parametrize("R,gamma,V,rank,wdt", SAMPLING_CASES)
def test_markov_sampling_and_rejection_verify(spec, ws, R, gamma, V, rank, wdt):
    wl = _wl(R, gamma, V, rank, wdt, seed=100 + V, T=0.8)
    g = to_dev(wl, "cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g.get("W1"), g.get("W2"), g["anchors"],
                                                 g["u_draft"], wl.temperature, rank=rank,
                                                 workspace=ws)
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, wl.temperature,
                                rank=rank)
    same = compare_proposals(toks, logp, stats, ref)
    assert same.mean() > 0.9
    for lengths in (None, torch.tensor([(3 * i) % (gamma + 1) for i in range(R)],
                                       dtype=torch.int32)):
        n, out, nxt = spec.spec_verify_rejection(
            g["target"], g["U"], g.get("W1"), g.get("W2"), g["anchors"], toks, logp, stats,
            g["u_accept"], g["u_resid"], wl.temperature,
            None if lengths is None else lengths.cuda(), rank=rank, workspace=ws)
        rv = oracle.verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, ref["tokens"],
                                     wl.u_accept, wl.u_resid, wl.temperature, lengths, rank=rank)
        gn, go, gx = n.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy()
        ok = same.copy()
        # near-tie acceptance decisions and final draws with a small CDF margin may differ
        compare_verify(gn, go, gx, rv, same)
        assert ((gn[ok] >= 0) & (gn[ok] <= (gamma if lengths is None else
                                             lengths.numpy()[ok]))).all()


def test_target_stats_match_oracle(spec, ws):
    wl = W.markov_rejection("cpu", R=5, gamma=2, V=20000, rank=64, seed=3, temperature=0.7)
    st = spec.spec_target_stats(wl.target.cuda(), 0.7, workspace=ws).cpu().numpy()
    for r in range(5):
        for i in range(3):
            p = oracle.target_probs(wl.target, r, i, 0.7)
            z = wl.target[r, i].double().numpy() * float(np.float32(1) / np.float32(0.7))
            m = z.max()
            lz = np.log(np.exp(z - m).sum())
            # the page's normaliser identity: p = exp(z - m - log Z)
            assert abs(np.exp(z[7] - m - lz) - p[7]) < 1e-12
            row = r * 3 + i
            assert abs((st[row, 0] + st[row, 1]) - (m + lz)) <= LOG_TOL * max(1, abs(m + lz))


@pytest.mark.parametrize("R,gamma,V,rank", [(70, 4, 1000, 256), (5, 3, 2048, 0), (4, 2, 777, 40),
                                           (96, 16, 129280, 256)])
def test_tv_confidence_and_survival(spec, ws, R, gamma, V, rank):
    wl = _wl(R, gamma, V, rank, "bf16", seed=200 + V, T=0.9)
    g = to_dev(wl, "cuda")
    toks = torch.randint(0, V, (R, gamma), generator=torch.Generator().manual_seed(1),
                         dtype=torch.int32)
    conf, surv = spec.spec_tv_confidence(g["U"], g["target"], g.get("W1"), g.get("W2"),
                                         g["anchors"], toks.cuda(), wl.temperature, rank=rank,
                                         workspace=ws)
    ref = oracle.tv_confidence(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, toks, wl.temperature,
                               rank=rank)
    assert_conf_close(conf, ref["conf"])
    assert_conf_close(surv, ref["survival"], "survival")
    s = surv.cpu().numpy()
    assert np.all(np.diff(s, axis=1) <= 0)


@pytest.mark.parametrize("R,gamma,kind", [(1, 1, 0), (3, 5, 1), (37, 7, 0), (512, 16, 1),
                                          (1024, 16, 2), (16384, 1, 0)])
def test_scheduler_bit_exact(spec, ws, R, gamma, kind):
    a = W.random_survival(R, gamma, seed=R + gamma)
    if kind == 2:
        a[:, :] = a[:, :1]                       # many equal survivals: tie order matters
    Bmax = R * (gamma + 1)
    if kind == 1:
        sps = W.sps_table(Bmax)
    else:
        sps = torch.from_numpy(np.random.default_rng(R).uniform(0.5, 1.0, Bmax + 1))
    lengths, B, theta = spec.spec_schedule_prefix(a.cuda(), sps.cuda(), workspace=ws)
    ref = oracle.schedule_prefix(a, sps.numpy())
    np.testing.assert_array_equal(lengths.cpu().numpy(), ref["lengths"])
    assert int(B.item()) == ref["B"]
    assert float(theta.item()) == ref["theta"]          # bit-identical


@pytest.mark.parametrize("R,gamma,kind", [(1, 1, 0), (37, 7, 0), (512, 16, 1), (1024, 16, 2),
                                          (16384, 1, 0)])
def test_scheduler_topk_bit_exact(spec, ws, R, gamma, kind):
    """Dynamic top-K: every capacity from below R to beyond Bmax, bit-exact against the oracle,
    and the fused Theta optimum equals the plain scheduler's."""
    a = W.random_survival(R, gamma, seed=7 * R + gamma)
    if kind == 2:
        a[:, :] = a[:, :1]
    Bmax = R * (gamma + 1) - (R // 3)
    sps = W.sps_table(Bmax) if kind == 1 else torch.from_numpy(
        np.random.default_rng(R + 1).uniform(0.5, 1.0, Bmax + 1))
    opt = oracle.schedule_prefix(a, sps.numpy())
    caps = sorted({-5, 0, R - 1, R, R + 1, (R + Bmax) // 2, opt["B"], Bmax, Bmax + 3})
    ad, sd = a.cuda(), sps.cuda()
    for cap in caps:
        c = torch.tensor([cap], dtype=torch.int32, device="cuda")
        b_opt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        lengths, B, theta = spec.spec_schedule_prefix(ad, sd, workspace=ws, capacity=c,
                                                      B_opt_out=b_opt)
        ref = oracle.schedule_topk(a, sps.numpy(), max(cap, 0))
        np.testing.assert_array_equal(lengths.cpu().numpy(), ref["lengths"])
        assert int(B.item()) == ref["B"]
        assert float(theta.item()) == ref["theta"]
        assert int(b_opt.item()) == opt["B"]
        st = spec.spec_device_status(ws)
        assert st == (spec.SPEC_DEV_BAD_LENGTH if cap < 0 else 0)


# ----------------------------------------------------------------------------- lossless grid

def test_rejection_pipeline_per_uniform_agreement_v8(spec, ws):
    """The whole GPU pipeline at V = 8, gamma = 2 on a stratified grid of uniforms, compared
    uniform by uniform with the oracle (whose output distribution is pinned by exact
    enumeration); the emitted first token's frequencies then follow the target."""
    R, gamma, V, rank, T = 4096, 2, 8, 64, 0.9
    gen = torch.Generator().manual_seed(77)
    U1 = torch.randn(1, gamma, V, generator=gen).mul(1.5)
    T1 = torch.randn(1, gamma + 1, V, generator=gen).mul(1.5)
    U = U1.expand(R, -1, -1).contiguous().to(torch.bfloat16)
    Tg = T1.expand(R, -1, -1).contiguous().to(torch.bfloat16)
    W1 = torch.randn(V, rank, generator=gen).mul(0.3).to(torch.bfloat16)
    W2 = torch.randn(V, rank, generator=gen).mul(0.3).to(torch.bfloat16)
    anchors = torch.full((R,), 2, dtype=torch.int32)
    strata = (torch.arange(R, dtype=torch.float64) + 0.5) / R
    perm = lambda s: strata[torch.randperm(R, generator=torch.Generator().manual_seed(s))]
    u_draft = torch.stack([perm(1), perm(2)], 1).float()
    u_acc = torch.stack([perm(3), perm(4)], 1).float()
    u_res = perm(5).float()
    d = lambda t: t.cuda()
    toks, logp, stats = spec.spec_markov_propose(d(U), d(W1), d(W2), d(anchors), d(u_draft), T,
                                                 workspace=ws)
    n, out, nxt = spec.spec_verify_rejection(d(Tg), d(U), d(W1), d(W2), d(anchors), toks, logp,
                                             stats, d(u_acc), d(u_res), T, workspace=ws)
    ref = oracle.markov_propose(U, W1, W2, anchors, u_draft, T)
    same = compare_proposals(toks, logp, stats, ref)
    rv = oracle.verify_rejection(Tg, U, W1, W2, anchors, ref["tokens"], u_acc, u_res, T)
    amb = (np.nan_to_num(rv["accept_margin"], nan=1.0) < 1e-6).any(axis=1) | (
        rv["resid_margin"] < 1e-6)
    go = out.cpu().numpy()
    agree = (go == rv["out_tokens"]).all(axis=1)
    assert (agree | amb | ~same).all()
    assert (agree & same).mean() > 0.99
    # first emitted token ~ target row 0 (the target here does not depend on the prefix)
    pt0 = oracle.target_probs(Tg, 0, 0, T)
    freq = np.bincount(go[:, 0], minlength=V) / R
    assert np.abs(freq - pt0).max() < 4.0 / np.sqrt(R)


# ----------------------------------------------------------------------------- device faults

def test_device_status_flags_bad_tokens_without_faulting(spec):
    ws = spec.Workspace(device="cuda")
    wl = W.markov_rejection("cpu", R=4, gamma=2, V=512, rank=64, seed=9)
    g = to_dev(wl, "cuda")
    g["anchors"][1] = 512                               # out of range
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"],
                                                 g["u_draft"], 1.0, workspace=ws)
    torch.cuda.synchronize()
    st = ws.status()
    assert st & spec.SPEC_DEV_BAD_TOKEN
    t = toks.cpu()
    assert ((t >= 0) & (t < 512)).all()
    assert ws.status() == 0                              # cleared by the previous read


def test_device_status_flags_nonfinite_logits(spec):
    ws = spec.Workspace(device="cuda")
    wl = W.markov_rejection("cpu", R=3, gamma=2, V=512, rank=0, seed=9)
    U = wl.U.clone()
    U[2, 0, :] = float("nan")
    toks, _, _ = spec.spec_markov_propose(U.cuda(), None, None, None, wl.u_draft.cuda(), 1.0,
                                          rank=0, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() & spec.SPEC_DEV_NONFINITE
    t = toks.cpu()
    assert ((t >= 0) & (t < 512)).all()


def test_greedy_bf16_markov_tensor_core(spec, ws):
    """Greedy proposals with bf16 weights (tensor-core bias). Reading: the bias is accumulated in
    fp32 in the tensor core's order, the oracle's exactly (products of bf16 values are exact and
    summed in fp64), and fp32 logits of magnitude ~8 round at ~1e-6; so an id may differ from
    the oracle's only where the oracle's top-two score gap is below 1e-6. Such cases are counted
    in the parity totals; every other request must be identical (later positions of a request
    that differed depend on a different token and are not compared)."""
    wl = W.markov_rejection("cpu", R=150, gamma=4, V=2056, rank=128, seed=31)
    wl.W1 = (wl.W1.float() * 20).to(torch.bfloat16)     # make the bias matter
    g = to_dev(wl, "cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"], None, 0.0,
                                                 workspace=ws)
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, None, 0.0)
    compare_proposals(toks, logp, stats, ref)      # the margin rule, with MARGIN = 1e-6
