"""Pins of the CPU oracle to what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: a worked example printed on
the pages (tests/golden), a closed form, an invariant, a special case that reduces to a library
routine, an exact enumeration, or brute force on tiny inputs.
"""
import itertools

import numpy as np
import pytest
import torch

from conftest import read_golden
from draft_sampling_verification_markov_gb300 import workloads as wlmod


def _bf16_bits(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


# --------------------------------------------------------------------------- softmax / sampling

def test_softmax_sums_to_one_and_is_shift_invariant(orc):
    rng = np.random.default_rng(0)
    for n in (1, 2, 8, 1000, 129280):
        z = rng.normal(0, 3, n)
        p, m, logz = orc.softmax(z)
        assert abs(p.sum() - 1.0) < 1e-12
        assert (p >= 0).all()
        p2, m2, logz2 = orc.softmax(z + 123.5)
        np.testing.assert_allclose(p2, p, rtol=1e-12, atol=1e-300)
        assert m2 == pytest.approx(m + 123.5)
        assert logz2 == pytest.approx(logz, abs=1e-12)
        # log-normaliser identity: log sum exp(z) = m + log Z
        zz = z - z.max()
        assert m + logz == pytest.approx(z.max() + np.log(np.exp(zz).sum()), rel=1e-12)


def test_softmax_matches_library_on_rank0_draft(orc):
    """rank 0 draft probabilities reduce to scipy's softmax of U * invT."""
    scipy_special = pytest.importorskip("scipy.special")
    U = torch.randn(2, 3, 50, generator=torch.Generator().manual_seed(3)) * 2
    p, _, _ = orc.draft_probs(U, None, None, r=1, k=2, prev=0, temperature=0.7, rank=0)
    invT = float(np.float32(1.0) / np.float32(0.7))
    ref = scipy_special.softmax(U[1, 1].double().numpy() * invT)
    np.testing.assert_allclose(p, ref, rtol=1e-12)


def test_sample_reproduces_distribution_by_counting(orc):
    rng = np.random.default_rng(1)
    p = rng.dirichlet(np.ones(8))
    N = 20000
    counts = np.zeros(8)
    for i in range(N):
        v, _ = orc.sample(p, (i + 0.5) / N)
        counts[v] += 1
    # every token receives the uniforms of its CDF interval: N * p(v) +- 1
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-9)


def test_sample_smallest_crossing_rule_and_zero_mass(orc):
    p = np.array([0.25, 0.0, 0.25, 0.5])
    assert orc.sample(p, 0.0)[0] == 0
    assert orc.sample(p, 0.2499)[0] == 0
    assert orc.sample(p, 0.25)[0] == 2          # C(0) = 0.25 is not > 0.25; p(1) = 0 skipped
    assert orc.sample(p, 0.49)[0] == 2          # C = [0.25, 0.25, 0.5, 1.0]
    assert orc.sample(p, 0.5)[0] == 3
    assert orc.sample(p, 0.999999)[0] == 3
    v, mrg = orc.sample(p, 0.3)
    assert v == 2 and mrg == pytest.approx(0.05)
    # one-hot: the same token for every u
    oh = np.zeros(16)
    oh[11] = 1.0
    assert {orc.sample(oh, u)[0] for u in np.linspace(0, 0.999, 50)} == {11}
    # rounding leaves no crossing: the largest positive-mass token is returned
    assert orc.sample(np.array([0.3, 0.3, 0.0]), 0.9)[0] == 1


def test_argmax_ties_go_to_lowest_index(orc):
    assert orc.argmax(np.array([1.0, 5.0, 5.0, 2.0]))[0] == 1
    assert orc.argmax(np.array([7.0, 7.0]))[0] == 0
    v, gap = orc.argmax(np.array([0.0, 3.0, 2.5]))
    assert v == 1 and gap == pytest.approx(0.5)


# --------------------------------------------------------------------------- greedy verify

def _onehot_rows(argmax_ids, V, dtype=torch.float32):
    t = torch.zeros(len(argmax_ids), V, dtype=torch.float32)
    for i, a in enumerate(argmax_ids):
        t[i, a] = 10.0
    return t.to(dtype)


def test_greedy_verify_worked_example(orc):
    g = read_golden("greedy_window_example.txt")
    ids = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in g["tokens"].split()}
    window = [ids[t] for t in g["window"].split()]
    rows = [ids[t] for t in g["target_argmax_rows"].split()]
    V = 8
    target = _onehot_rows(rows, V, torch.bfloat16).unsqueeze(0)       # [1, gamma+1, V]
    drafts = np.array([window[1:]], dtype=np.int32)                   # [1, gamma]
    out = orc.verify_greedy(target, drafts)
    assert out["accept_len"][0] == int(g["expected_accept_len"])
    exp_out = [ids[t] for t in g["expected_out"].split()]
    assert list(out["out_tokens"][0][:len(exp_out)]) == exp_out
    assert out["next_anchor"][0] == ids[g["expected_next_anchor"]]


def test_greedy_verify_window_counting(orc):
    g = read_golden("window_counting.txt")
    gamma = int(g["num_steps"])
    assert gamma + 1 == int(g["window_width"])
    V = 16
    drafts = np.array([[3, 5, 7], [3, 5, 7], [3, 5, 7]], dtype=np.int32)
    all_match = _onehot_rows([3, 5, 7, 9], V)
    first_miss = _onehot_rows([4, 5, 7, 9], V)
    second_miss = _onehot_rows([3, 6, 7, 9], V)
    target = torch.stack([all_match, first_miss, second_miss])
    out = orc.verify_greedy(target, drafts)
    emitted = (out["out_tokens"] >= 0).sum(axis=1)
    assert emitted[0] == int(g["all_accepted_emitted"])
    assert list(out["out_tokens"][0]) == [3, 5, 7, 9]
    assert emitted[1] == int(g["first_rejected_emitted"])
    assert list(out["out_tokens"][1]) == [4, -1, -1, -1]
    assert list(out["out_tokens"][2]) == [3, 6, -1, -1]
    assert list(out["accept_len"]) == [3, 0, 1]
    assert list(out["next_anchor"]) == [9, 4, 6]


def test_greedy_verify_respects_lengths(orc):
    V = 16
    drafts = np.array([[3, 5, 7]] * 3, dtype=np.int32)
    target = torch.stack([_onehot_rows([3, 5, 7, 9], V)] * 3)
    out = orc.verify_greedy(target, drafts, lengths=np.array([0, 2, 3], dtype=np.int32))
    assert list(out["accept_len"]) == [0, 2, 3]
    assert list(out["out_tokens"][0]) == [3, -1, -1, -1]       # bonus from row 0
    assert list(out["out_tokens"][1]) == [3, 5, 7, -1]         # x1, x2, bonus = argmax row 2
    assert list(out["next_anchor"]) == [3, 7, 9]


# --------------------------------------------------------------------------- Markov head

def test_markov_bias_exact_integer_case_matches_matmul(orc):
    """With small-integer fp32 values every fp32 operation is exact, so the biased scores are
    the integer matrix product U + W1[prev] @ W2^T (reduces to numpy's matmul)."""
    rng = np.random.default_rng(5)
    R, gamma, V, rank = 2, 3, 12, 5
    U = rng.integers(-20, 20, (R, gamma, V)).astype(np.float32)
    W1 = rng.integers(-3, 4, (V, rank)).astype(np.float32)
    W2 = rng.integers(-3, 4, (V, rank)).astype(np.float32)
    anchors = np.array([4, 9], dtype=np.int32)
    out = orc.markov_propose(U, W1, W2, anchors, None, 0.0)
    prev = anchors.copy()
    for k in range(gamma):
        s = U[:, k, :].astype(np.int64) + W1[prev].astype(np.int64) @ W2.T.astype(np.int64)
        want = np.argmax(s, axis=1)          # numpy breaks ties to the lowest index too
        assert list(out["tokens"][:, k]) == list(want)
        prev = want.astype(np.int32)
    # greedy log-probs are those of the unscaled softmax of the scores
    s0 = U[:, 0, :].astype(np.float64) + W1[anchors].astype(np.float64) @ W2.T
    lse = np.log(np.exp(s0 - s0.max(1, keepdims=True)).sum(1)) + s0.max(1)
    np.testing.assert_allclose(out["logp"][:, 0], s0[np.arange(R), out["tokens"][:, 0]] - lse,
                               rtol=0, atol=1e-12)


def test_markov_head_follows_planted_transition_chain(orc):
    """A bias that makes token f(prev) dominate must drive greedy proposals along the chain
    prev -> f(prev), starting from the anchor at position 1 (anchor-first layout)."""
    V, rank, R, gamma = 32, 32, 3, 6
    f = np.array([(7 * v + 3) % V for v in range(V)])
    W1 = np.eye(V, rank, dtype=np.float32)                 # W1[x] = e_x
    W2 = np.zeros((V, rank), dtype=np.float32)
    for x in range(V):
        W2[f[x], x] = 50.0                                 # row f(x) projects onto e_x
    U = np.random.default_rng(2).normal(0, 1, (R, gamma, V)).astype(np.float32)
    anchors = np.array([0, 5, 31], dtype=np.int32)
    for dtype in ("f32", "bf16"):
        if dtype == "bf16":
            args = [_bf16_bits(a) for a in (U, W1, W2)]
        else:
            args = [U, W1, W2]
        out = orc.markov_propose(*args, anchors, None, 0.0)
        for r in range(R):
            chain, x = [], anchors[r]
            for _ in range(gamma):
                x = f[x]
                chain.append(x)
            assert list(out["tokens"][r]) == chain, dtype


def test_zero_projection_reduces_to_plain_draft(orc):
    rng = torch.Generator().manual_seed(9)
    R, gamma, V, rank = 3, 4, 300, 16
    U = (torch.randn(R, gamma, V, generator=rng) * 2).to(torch.bfloat16)
    W1 = (torch.randn(V, rank, generator=rng)).to(torch.bfloat16)
    W2 = torch.zeros(V, rank, dtype=torch.bfloat16)
    anchors = torch.tensor([1, 2, 3], dtype=torch.int32)
    u = torch.rand(R, gamma, generator=rng)
    a = orc.markov_propose(U, W1, W2, anchors, u, 0.8)
    b = orc.markov_propose(U, None, None, anchors, u, 0.8)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_allclose(a["logp"], b["logp"], rtol=0, atol=0)
    # the sampled token carries the logged probability
    for r in range(R):
        for k in range(gamma):
            p, _, _ = orc.draft_probs(U, None, None, r, k + 1, 0, 0.8, rank=0)
            assert np.log(p[a["tokens"][r, k]]) == pytest.approx(a["logp"][r, k], rel=1e-12)


def test_propose_sampling_frequencies_match_probabilities(orc):
    """Sweeping the draft uniform over a fine grid reproduces p_d at position 1 by counting."""
    rng = torch.Generator().manual_seed(4)
    V, rank, N = 8, 4, 4000
    U = torch.randn(N, 1, V, generator=rng).mul(1.5).to(torch.bfloat16)
    U[:] = U[0]                                     # every request sees the same logits
    W1 = torch.randn(V, rank, generator=rng).to(torch.bfloat16)
    W2 = torch.randn(V, rank, generator=rng).to(torch.bfloat16)
    anchors = torch.full((N,), 5, dtype=torch.int32)
    u = ((torch.arange(N, dtype=torch.float64) + 0.5) / N).float().reshape(N, 1)
    out = orc.markov_propose(U, W1, W2, anchors, u, 1.3)
    p, _, _ = orc.draft_probs(U, W1, W2, 0, 1, 5, 1.3)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-6)


# --------------------------------------------------------------------------- rejection verify

def test_identical_distributions_accept_every_token(orc):
    """p_d == p_t (zero projection, target rows equal to the draft rows) accepts all proposed
    tokens for every u_accept < 1; the output token is then drawn from target row gamma."""
    rng = torch.Generator().manual_seed(11)
    R, gamma, V, rank = 16, 5, 64, 8
    U = torch.randn(R, gamma, V, generator=rng).mul(2).to(torch.bfloat16)
    target = torch.cat([U, torch.randn(R, 1, V, generator=rng).to(torch.bfloat16)], dim=1)
    W1 = torch.randn(V, rank, generator=rng).to(torch.bfloat16)
    W2 = torch.zeros(V, rank, dtype=torch.bfloat16)
    anchors = torch.randint(0, V, (R,), generator=rng, dtype=torch.int32)
    prop = orc.markov_propose(U, W1, W2, anchors, torch.rand(R, gamma, generator=rng), 0.9)
    u_acc = torch.rand(R, gamma, generator=rng)
    u_acc[0] = float(np.nextafter(np.float32(1), np.float32(0)))    # the largest u < 1
    u_res = torch.rand(R, generator=rng)
    out = orc.verify_rejection(target, U, W1, W2, anchors, prop["tokens"], u_acc, u_res, 0.9)
    assert (out["accept_len"] == gamma).all()
    for r in range(R):
        pt = orc.target_probs(target, r, gamma, 0.9)
        assert out["out_tokens"][r, gamma] == orc.sample(pt, float(u_res[r]))[0]


def test_accept_test_realises_min_ratio(orc):
    rng = np.random.default_rng(8)
    for _ in range(200):
        pd, pt = rng.uniform(1e-6, 1, 2)
        a = orc.accept_prob(pd, pt)
        assert a == pytest.approx(min(1.0, pt / pd), rel=1e-15)
        if a < 1.0:
            assert orc.accept_test(a * (1 - 1e-9), pd, pt)
            assert not orc.accept_test(a * (1 + 1e-9), pd, pt)
        else:
            assert orc.accept_test(1 - 1e-12, pd, pt)
    assert orc.accept_test(0.0, 0.3, 1e-300)       # u = 0 always accepts


def test_residual_is_normalised_positive_part(orc):
    rng = np.random.default_rng(12)
    pt, pd = rng.dirichlet(np.ones(10)), rng.dirichlet(np.ones(10))
    q, z = orc.residual(pt, pd)
    assert abs(q.sum() - 1) < 1e-12 and (q >= 0).all()
    # mass only where the target exceeds the draft
    assert np.all((q > 0) == (pt > pd))
    # the normaliser equals the total variation distance 1/2 ||pt - pd||_1
    assert z == pytest.approx(0.5 * np.abs(pt - pd).sum(), rel=1e-12)


def _enumeration_problem(seed, gamma, V=8, rank=4, temperature=0.8):
    g = torch.Generator().manual_seed(seed)
    U = torch.randn(1, gamma, V, generator=g).mul(1.5).to(torch.bfloat16)
    W1 = torch.randn(V, rank, generator=g).to(torch.bfloat16)
    W2 = torch.randn(V, rank, generator=g).to(torch.bfloat16)
    Tb = torch.randn(gamma + 1, V, generator=g).mul(1.5)          # target base rows
    M = torch.randn(V, V, generator=g)                            # target transition table
    anchor = 3
    return U, W1, W2, Tb, M, anchor, temperature


def _target_for(Tb, M, prefix):
    """Prefix-dependent target logits: row i = Tb[i] + M[prefix[i]] (prefix[0] = anchor)."""
    rows = torch.stack([Tb[i] + M[prefix[i]] for i in range(len(prefix))])
    return rows.to(torch.bfloat16).unsqueeze(0)


@pytest.mark.parametrize("gamma,top_k", [(1, None), (2, None), (3, None), (2, 3), (3, 3)])
def test_rejection_sampling_is_lossless_by_exact_enumeration(orc, gamma, top_k):
    """Sum exactly over every draft sequence, every accept/reject branch and every final token;
    the emitted block, padded with fresh target draws, must follow the target chain rule
    P(y_1..y_{gamma+1}) = prod_i p_t(y_{i+1} | y_i) (y_0 = anchor). Draft and target are both
    prefix-dependent (a Markov head on the draft side, a transition table on the target side)
    and share the temperature. With top_k, every target row keeps only its 3 largest logits
    (the others are -inf): draft tokens outside that nucleus must never survive, and the
    emitted block must still follow the truncated target chain."""
    from draft_sampling_verification_markov_gb300.workloads import truncate_rows
    U, W1, W2, Tb, M, anchor, T = _enumeration_problem(100 + gamma, gamma)
    V = U.shape[-1]
    # target row i conditioned on the token at window position i
    tp = np.zeros((gamma + 1, V, V))
    for prev in range(V):
        tgt = _target_for(Tb, M, [prev] * (gamma + 1))
        if top_k is not None:
            tgt = truncate_rows(tgt, top_k=top_k)
        for i in range(gamma + 1):
            tp[i, prev] = orc.target_probs(tgt, 0, i, T)
            if top_k is not None:
                assert np.count_nonzero(tp[i, prev]) == top_k
    # draft position k conditioned on the previous token
    pd = np.zeros((gamma + 1, V, V))
    for k in range(1, gamma + 1):
        for prev in range(V):
            pd[k, prev] = orc.draft_probs(U, W1, W2, 0, k, prev, T)[0]

    def pad_after(L, y):
        """distribution of (y_{L+1}..y_{gamma+1}) given y_L = y under the target chain."""
        if L == gamma + 1:
            return np.array(1.0)
        return np.stack([tp[L, y, v] * pad_after(L + 1, v) for v in range(V)])

    P = np.zeros((V,) * (gamma + 1))
    for x in itertools.product(range(V), repeat=gamma):
        prefix = (anchor,) + x
        reach = 1.0
        for k in range(1, gamma + 1):
            reach *= pd[k, prefix[k - 1], x[k - 1]]
        for n in range(gamma + 1):
            if n < gamma:
                # position n+1 is tested against target row n, both conditioned on x_n
                p_t, p_d = tp[n, prefix[n]], pd[n + 1, prefix[n]]
                alpha = orc.accept_prob(p_d[x[n]], p_t[x[n]])
                q, _ = orc.residual(p_t, p_d)
                w = reach * (1.0 - alpha)
                reach *= alpha
            else:
                q, w = tp[gamma, prefix[gamma]], reach
            if w <= 0:
                continue
            for y in range(V):
                if q[y] > 0:
                    P[x[:n] + (y,)] += w * q[y] * pad_after(n + 1, y)
    want = pad_after(0, anchor)
    assert abs(P.sum() - 1.0) < 1e-12
    assert np.max(np.abs(P - want)) <= 1e-12


def test_uniform_driven_verify_matches_branch_probabilities(orc):
    """The uniform-driven verify realises the branch probabilities used above: sweeping
    u_accept at position 1 accepts exactly below alpha, and sweeping u_resid reproduces the
    residual distribution by counting."""
    U, W1, W2, Tb, M, anchor, T = _enumeration_problem(7, 1)
    V = U.shape[-1]
    pd, _, _ = orc.draft_probs(U, W1, W2, 0, 1, anchor, T)
    tgt = _target_for(Tb, M, [anchor, 0])
    pt = orc.target_probs(tgt, 0, 0, T)          # row 0 depends on the anchor only
    x1 = int(np.argmax(pd - pt))                 # a token the draft over-proposes
    tgt = _target_for(Tb, M, [anchor, x1])
    alpha = orc.accept_prob(pd[x1], pt[x1])
    assert alpha < 1.0
    q, _ = orc.residual(pt, pd)
    N = 4000
    uu = ((np.arange(N) + 0.5) / N).astype(np.float32)
    counts = np.zeros(V)
    accepted = 0
    for i in range(N):
        for ua, ur in ((uu[i], 0.5), (0.999999, uu[i])):
            out = orc.verify_rejection(tgt, U, W1, W2, np.array([anchor], np.int32),
                                       np.array([[x1]], np.int32), np.array([[ua]], np.float32),
                                       np.array([ur], np.float32), T)
            if ua != 0.999999:
                accepted += int(out["accept_len"][0] == 1)
            else:
                counts[out["out_tokens"][0, 0]] += 1
    assert abs(accepted - N * alpha) <= 1.0
    assert np.all(np.abs(counts - N * q) <= 1.0 + 1e-6)


# --------------------------------------------------------------------------- confidence

def test_tv_confidence_pins(orc):
    g = torch.Generator().manual_seed(21)
    R, gamma, V, rank = 4, 4, 40, 8
    U = torch.randn(R, gamma, V, generator=g).mul(2).to(torch.bfloat16)
    W1 = torch.randn(V, rank, generator=g).mul(0.3).to(torch.bfloat16)
    W2 = torch.randn(V, rank, generator=g).mul(0.3).to(torch.bfloat16)
    target = torch.randn(R, gamma + 1, V, generator=g).mul(2).to(torch.bfloat16)
    anchors = torch.randint(0, V, (R,), generator=g, dtype=torch.int32)
    drafts = torch.randint(0, V, (R, gamma), generator=g, dtype=torch.int32)
    out = orc.tv_confidence(U, target, W1, W2, anchors, drafts, 0.9)
    c, a = out["conf"], out["survival"]
    assert np.all((c > 0) & (c <= 1))
    # survival: running product, non-increasing
    np.testing.assert_allclose(a, np.cumprod(c, axis=1), rtol=1e-14)
    assert np.all(np.diff(a, axis=1) <= 0)
    for r in range(R):
        prev = int(anchors[r])
        for k in range(1, gamma + 1):
            pd, _, _ = orc.draft_probs(U, W1, W2, r, k, prev, 0.9)
            pt = orc.target_probs(target, r, k - 1, 0.9)
            # the page's form 1 - 1/2 ||p_d - p_t||_1
            assert c[r, k - 1] == pytest.approx(1 - 0.5 * np.abs(pd - pt).sum(), abs=1e-13)
            # and the exact acceptance probability of the proposed position
            acc = sum(pd[v] * orc.accept_prob(pd[v], pt[v]) for v in range(V))
            assert c[r, k - 1] == pytest.approx(acc, abs=1e-13)
            prev = int(drafts[r, k - 1])


def test_tv_confidence_extremes(orc):
    V, gamma = 16, 2
    U = torch.full((2, gamma, V), -60.0)
    target = torch.full((2, gamma + 1, V), -60.0)
    U[0, :, 3] = 60.0
    target[0, :gamma, 3] = 60.0            # identical one-hots -> c* = 1
    U[1, :, 3] = 60.0
    target[1, :gamma, 4] = 60.0            # disjoint one-hots -> c* = 0
    out = orc.tv_confidence(U, target, None, None, None,
                            np.zeros((2, gamma), np.int32), 1.0, rank=0)
    assert np.allclose(out["conf"][0], 1.0, atol=1e-15)
    assert np.all(out["conf"][1] < 1e-40)
    # identical distributions in general: c* = 1
    g = torch.Generator().manual_seed(2)
    Ur = torch.randn(3, gamma, V, generator=g)
    Tr = torch.cat([Ur, torch.randn(3, 1, V, generator=g)], dim=1)
    out = orc.tv_confidence(Ur, Tr, None, None, None, np.zeros((3, gamma), np.int32), 0.6,
                            rank=0)
    assert np.allclose(out["conf"], 1.0, atol=1e-14)


# --------------------------------------------------------------------------- scheduler

def _brute_force(a, sps):
    R, gamma = a.shape
    best, arg = -1.0, []
    for ls in itertools.product(range(gamma + 1), repeat=R):
        B = sum(1 + l for l in ls)
        if B >= len(sps):
            continue
        tau = sum(1.0 + sum(float(a[r, j]) for j in range(ls[r])) for r in range(R))
        th = tau * sps[B]
        if th > best * (1 + 1e-12):
            best, arg = th, [ls]
        elif th >= best * (1 - 1e-12):
            arg.append(ls)
    return best, arg


def _theta(a, sps, ls):
    B = sum(1 + l for l in ls)
    tau = sum(1.0 + sum(float(a[r, j]) for j in range(ls[r])) for r in range(len(ls)))
    return tau * sps[B]


@pytest.mark.parametrize("seed", range(12))
def test_scheduler_matches_brute_force(orc, seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 5))
    gamma = int(rng.integers(1, 6))
    a = wlmod.random_survival(R, gamma, seed=seed).numpy()
    Bmax = R * (gamma + 1) + int(rng.integers(-R * gamma // 2, 3))
    Bmax = max(Bmax, R)
    kind = seed % 3
    if kind == 0:
        sps = rng.uniform(0.1, 1.0, Bmax + 1)                        # arbitrary profile
    elif kind == 1:
        sps = wlmod.sps_table(Bmax, base_ms=1.0, step_ms=0.7, step=3).numpy()   # sawtooth
    else:
        sps = 1.0 / (1.0 + 0.3 * np.arange(Bmax + 1))                 # smooth decreasing
    out = orc.schedule_prefix(a, sps)
    best, argset = _brute_force(a, sps)
    assert out["theta"] == pytest.approx(best, rel=1e-9)
    ls = tuple(int(x) for x in out["lengths"])
    assert _theta(a, sps, ls) >= best * (1 - 1e-9)
    assert out["B"] == sum(1 + l for l in ls)


def test_scheduler_special_cases(orc):
    a = wlmod.random_survival(3, 4, seed=5).numpy()
    # constant SPS: more verified tokens always raise tau -> verify everything
    out = orc.schedule_prefix(a, np.full(3 * 5 + 1, 2.0))
    assert list(out["lengths"]) == [4, 4, 4] and out["B"] == 15
    assert out["theta"] == pytest.approx(2.0 * (3 + a.astype(np.float64).sum()), rel=1e-9)
    # SPS zero beyond B = R: verify nothing
    sps = np.zeros(16)
    sps[3] = 1.0
    out = orc.schedule_prefix(a, sps)
    assert list(out["lengths"]) == [0, 0, 0] and out["B"] == 3
    # equal survivals: the tie order is r ascending, then j ascending
    eq = np.full((2, 4), 0.5, dtype=np.float32)
    sps = np.zeros(2 * 5 + 1)
    sps[2:6] = 1.0                          # best is the largest K with B <= 5, i.e. K = 3
    out = orc.schedule_prefix(eq, sps)
    assert list(out["lengths"]) == [3, 0] and out["B"] == 5
    # Bmax below R * (gamma + 1) caps K
    out = orc.schedule_prefix(a, np.full(5, 1.0))
    assert out["B"] == 4 and sum(out["lengths"]) == 1
    # prefix closure under the tie order: equal values within a row stay in order
    eq2 = np.array([[1.0, 1.0, 1.0]], dtype=np.float32)
    sps = np.array([0, 1.0, 1.0, 1.0, 0.0])
    out = orc.schedule_prefix(eq2, sps)
    assert list(out["lengths"]) == [2]


# ----------------------------------------------------------------------------- grammar masks

def _bits(allowed_rows, V):
    """bool [R, V] -> uint32 words [R, ceil(V/32)], bit v%32 of word v/32."""
    R = len(allowed_rows)
    words = np.zeros((R, (V + 31) // 32), dtype=np.uint32)
    for r, row in enumerate(allowed_rows):
        for v in np.nonzero(row)[0]:
            words[r, v // 32] |= np.uint32(1 << (v % 32))
    return words


def test_masked_draft_is_the_renormalised_restriction(orc):
    g = torch.Generator().manual_seed(21)
    R, gamma, V, rank = 2, 2, 70, 8
    U = torch.randn(R, gamma, V, generator=g).mul(2).to(torch.bfloat16)
    W1 = torch.randn(V, rank, generator=g).mul(0.3).to(torch.bfloat16)
    W2 = torch.randn(V, rank, generator=g).mul(0.3).to(torch.bfloat16)
    allowed = np.random.default_rng(3).random((R, V)) < 0.4
    mask = _bits(allowed, V)
    for r in range(R):
        for k in (1, 2):
            p, _, _ = orc.draft_probs(U, W1, W2, r, k, 5, 0.8)
            pm, _, _ = orc.draft_probs(U, W1, W2, r, k, 5, 0.8, mask=mask)
            want = np.where(allowed[r], p, 0.0)
            np.testing.assert_allclose(pm, want / want.sum(), rtol=1e-12, atol=1e-300)
    ones = _bits(np.ones((R, V), bool), V)
    p1, _, _ = orc.draft_probs(U, W1, W2, 1, 2, 7, 0.8, mask=ones)
    p0, _, _ = orc.draft_probs(U, W1, W2, 1, 2, 7, 0.8)
    assert np.array_equal(p1, p0)


def test_masked_greedy_is_argmax_over_allowed_tokens(orc):
    """Small-integer fp32 values: the scores are the exact integer matrix product, so the
    masked argmax is checked by brute force (ties to the lowest allowed id)."""
    rng = np.random.default_rng(8)
    R, gamma, V, rank = 3, 4, 40, 6
    U = rng.integers(-6, 6, (R, gamma, V)).astype(np.float32)
    W1 = rng.integers(-2, 3, (V, rank)).astype(np.float32)
    W2 = rng.integers(-2, 3, (V, rank)).astype(np.float32)
    anchors = rng.integers(0, V, R).astype(np.int32)
    allowed = rng.random((R, V)) < 0.3
    allowed[:, 0] = True
    ref = orc.markov_propose(U, W1, W2, anchors, None, 0.0, mask=_bits(allowed, V))
    for r in range(R):
        prev = anchors[r]
        for k in range(gamma):
            s = U[r, k] + W1[prev] @ W2.T
            s = np.where(allowed[r], s, -np.inf)
            x = int(np.argmax(s))                     # numpy: first maximum
            assert ref["tokens"][r, k] == x
            prev = x


def test_masked_sampling_stays_in_the_allowed_set(orc):
    g = torch.Generator().manual_seed(5)
    R, gamma, V, rank = 64, 3, 50, 8
    U = torch.randn(R, gamma, V, generator=g).mul(2).to(torch.bfloat16)
    W1 = torch.randn(V, rank, generator=g).mul(0.3).to(torch.bfloat16)
    W2 = torch.randn(V, rank, generator=g).mul(0.3).to(torch.bfloat16)
    anchors = torch.randint(0, V, (R,), generator=g, dtype=torch.int32)
    u = torch.rand(R, gamma, generator=g)
    allowed = np.random.default_rng(9).random((R, V)) < 0.2
    allowed[:, 3] = True
    ref = orc.markov_propose(U, W1, W2, anchors, u, 0.9, mask=_bits(allowed, V))
    assert all(allowed[r, ref["tokens"][r, k]] for r in range(R) for k in range(gamma))


def test_masked_draft_rejection_is_lossless_by_exact_enumeration(orc):
    """The enumeration of the lossless pin with a draft restricted to 5 of 8 tokens: tokens the
    draft cannot propose still reach the output through the residual, and the emitted block
    follows the (unmasked) target chain."""
    gamma = 2
    U, W1, W2, Tb, M, anchor, T = _enumeration_problem(202, gamma)
    V = U.shape[-1]
    allowed = np.array([[1, 0, 1, 1, 0, 1, 0, 1]], bool)
    mask = _bits(allowed, V)
    tp = np.zeros((gamma + 1, V, V))
    for prev in range(V):
        tgt = _target_for(Tb, M, [prev] * (gamma + 1))
        for i in range(gamma + 1):
            tp[i, prev] = orc.target_probs(tgt, 0, i, T)
    pd = np.zeros((gamma + 1, V, V))
    for k in range(1, gamma + 1):
        for prev in range(V):
            pd[k, prev] = orc.draft_probs(U, W1, W2, 0, k, prev, T, mask=mask)[0]
            assert np.all(pd[k, prev][~allowed[0]] == 0)

    def pad_after(L, y):
        if L == gamma + 1:
            return np.array(1.0)
        return np.stack([tp[L, y, v] * pad_after(L + 1, v) for v in range(V)])

    P = np.zeros((V,) * (gamma + 1))
    for x in itertools.product(range(V), repeat=gamma):
        prefix = (anchor,) + x
        reach = 1.0
        for k in range(1, gamma + 1):
            reach *= pd[k, prefix[k - 1], x[k - 1]]
        if reach == 0:
            continue
        for n in range(gamma + 1):
            if n < gamma:
                p_t, p_d = tp[n, prefix[n]], pd[n + 1, prefix[n]]
                alpha = orc.accept_prob(p_d[x[n]], p_t[x[n]])
                q, _ = orc.residual(p_t, p_d)
                w = reach * (1.0 - alpha)
                reach *= alpha
            else:
                q, w = tp[gamma, prefix[gamma]], reach
            if w <= 0:
                continue
            for y in range(V):
                if q[y] > 0:
                    P[x[:n] + (y,)] += w * q[y] * pad_after(n + 1, y)
    want = pad_after(0, anchor)
    assert np.max(np.abs(P - want)) <= 1e-12


# ----------------------------------------------------------------------------- dynamic top-K

@pytest.mark.parametrize("seed", range(4))
def test_topk_takes_the_k_largest_survivals_prefix_closed(orc, seed):
    """Dynamic top-K (DSpark section 7): with capacity B the selected candidates are exactly the
    B - R largest survivals in queue order (a desc, r asc, j asc), prefix-closed per request;
    with the Theta-optimal B it reproduces the Theta scheduler."""
    rng = np.random.default_rng(50 + seed)
    R, gamma = 6, 5
    a = np.sort(rng.uniform(0.05, 1.0, (R, gamma)), axis=1)[:, ::-1].astype(np.float32)
    if seed == 3:
        a[:, :] = a[:, :1]                                  # ties: queue order decides
    sps = np.random.default_rng(seed).uniform(0.5, 1.0, R * (gamma + 1) + 1)
    order = sorted(((-float(a[r, j]), r, j) for r in range(R) for j in range(gamma)))
    for cap in (R - 3, R, R + 1, R + 7, R + R * gamma, R + R * gamma + 9):
        out = orc.schedule_topk(a, sps, cap)
        K = max(0, min(cap - R, R * gamma))
        want = np.zeros(R, dtype=np.int32)
        for _, r, j in order[:K]:
            want[r] += 1
        np.testing.assert_array_equal(out["lengths"], want)
        assert out["B"] == R + K
    opt = orc.schedule_prefix(a, sps)
    same = orc.schedule_topk(a, sps, opt["B"])
    np.testing.assert_array_equal(same["lengths"], opt["lengths"])
    assert same["theta"] == opt["theta"]


# ----------------------------------------------------------------------------- flattened batch

def test_flat_layout_worked_example(orc):
    """Packed rows of a variable-length verify batch (DSpark section 7), written out by hand for
    lengths (2, 0, 3) with gamma = 3: request 0 owns rows 0-2, request 1 row 3, request 2 rows
    4-7, and the last four of the 12 rows are past the batch."""
    out = orc.flat_layout(np.array([2, 0, 3]), 3)
    np.testing.assert_array_equal(out["offsets"], [0, 3, 4, 8])
    np.testing.assert_array_equal(out["row_req"], [0, 0, 0, 1, 2, 2, 2, 2, -1, -1, -1, -1])
    np.testing.assert_array_equal(out["row_pos"], [0, 1, 2, 0, 0, 1, 2, 3, -1, -1, -1, -1])


def test_flat_layout_batch_is_the_schedulers_B(orc):
    """The packed batch of the scheduler's lengths has exactly B = sum_r (1 + l_r) rows
    (DSpark section 6), and packing then reading row offsets[r] + i returns position (r, i)."""
    rng = np.random.default_rng(8)
    R, gamma = 23, 6
    a = np.sort(rng.uniform(0.0, 1.0, (R, gamma)), axis=1)[:, ::-1].astype(np.float32)
    sps = np.linspace(1.0, 0.4, R * (gamma + 1) + 1)
    sch = orc.schedule_prefix(a, sps)
    lay = orc.flat_layout(sch["lengths"], gamma)
    assert lay["offsets"][-1] == sch["B"]
    padded = rng.integers(0, 1 << 30, (R, gamma + 1))
    packed = np.full(R * (gamma + 1), -7)
    for r in range(R):
        for i in range(sch["lengths"][r] + 1):
            packed[lay["offsets"][r] + i] = padded[r, i]
    live = lay["row_req"] >= 0
    assert live.sum() == sch["B"]
    np.testing.assert_array_equal(packed[live], padded[lay["row_req"][live], lay["row_pos"][live]])
    assert (packed[~live] == -7).all()
