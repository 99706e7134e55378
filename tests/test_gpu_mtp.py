"""spec_mtp_greedy: the MTP/NextN greedy proposal and greedy verification in two chained
launches ("Module deepseek_v4_mtp", Forward; "DeepSeek-V4 MTP/NextN 怎样逐步生成候选", sections 三 and
四), against the oracle and, bit for bit, against the two-call form (spec_markov_propose at
rank 0, T = 0, then spec_verify_greedy) on the same bytes."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W

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


def _two_call(spec, D, T, lengths, ws):
    toks = spec.spec_markov_propose(D, None, None, None, None, 0.0, workspace=ws)[0] \
        if D is not None and D.shape[1] > 0 else torch.empty(T.shape[0], 0, dtype=torch.int32,
                                                             device=T.device)
    n, out, nxt = spec.spec_verify_greedy(T, toks, lengths, workspace=ws)
    return toks, n, out, nxt


def _check_oracle(D, T, lengths, got):
    toks, n, out, nxt = (x.cpu().numpy() for x in got)
    ref = oracle.markov_propose(D.cpu(), None, None, None, None, 0.0)
    np.testing.assert_array_equal(toks, ref["tokens"])
    rv = oracle.verify_greedy(T.cpu(), ref["tokens"], None if lengths is None else lengths.cpu())
    np.testing.assert_array_equal(n, rv["accept_len"])
    np.testing.assert_array_equal(out, rv["out_tokens"])
    np.testing.assert_array_equal(nxt, rv["next_anchor"])


def test_mtp_workload_at_its_size(spec, ws):
    """R = 64, gamma = 3, V = 129280 bf16 (the MTP-1 workload): oracle and two-call form."""
    wl = W.mtp_greedy("cuda", R=64, gamma=3, V=129280, seed=1002)
    got = spec.spec_mtp_greedy(wl.U, wl.target, workspace=ws)
    torch.cuda.synchronize()
    _check_oracle(wl.U, wl.target, None, got)
    np.testing.assert_array_equal(got[0].cpu().numpy(), wl.extra["planted_tokens"].cpu().numpy())
    ref = _two_call(spec, wl.U, wl.target, None, ws)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,gamma,V", [(37, 4, 20000), (5, 2, 8200), (3, 1, 8192), (2, 3, 16)])
def test_ties_lengths_and_ragged_chunks(spec, ws, dtype, R, gamma, V):
    """Logits drawn from a handful of integer values (many ties, which go to the lowest id),
    rows spanning several 4096-element chunks with a ragged last one, per-request lengths;
    target rows copy the draft argmax with probability 3/4 so that prefixes get accepted."""
    g = torch.Generator().manual_seed(R * 1000 + V)
    D = torch.randint(-3, 4, (R, gamma, V), generator=g).to(dtype)
    T = torch.randint(-3, 4, (R, gamma + 1, V), generator=g).to(dtype)
    # plant some draft argmaxes into the target rows before them
    x = D.float().argmax(dim=2)
    keep = torch.rand(R, gamma, generator=g) < 0.75
    for r in range(R):
        for k in range(gamma):
            if keep[r, k]:
                T[r, k, x[r, k]] = 9.0
    lengths = torch.randint(0, gamma + 1, (R,), generator=g, dtype=torch.int32)
    Dd, Td = D.cuda(), T.cuda()
    for ln in (None, lengths.cuda()):
        got = spec.spec_mtp_greedy(Dd, Td, ln, workspace=ws)
        torch.cuda.synchronize()
        _check_oracle(D, T, None if ln is None else lengths, got)
        ref = _two_call(spec, Dd, Td, ln, ws)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_unaligned_vocabulary_takes_the_two_call_form(spec, ws):
    """V = 1003 (rows not on 16-byte boundaries): the same results through the two calls."""
    wl = W.mtp_greedy("cpu", R=9, gamma=3, V=1003, seed=7)
    D, T = wl.U.cuda(), wl.target.cuda()
    got = spec.spec_mtp_greedy(D, T, workspace=ws)
    torch.cuda.synchronize()
    _check_oracle(wl.U, wl.target, None, got)


def test_no_draft_positions(spec, ws):
    """gamma = 0: the window is the bonus row alone; D is not read."""
    T = torch.randn(6, 1, 5000, dtype=torch.bfloat16)
    got = spec.spec_mtp_greedy(None, T.cuda(), workspace=ws)
    torch.cuda.synchronize()
    toks, n, out, nxt = (x.cpu() for x in got)
    assert toks.shape == (6, 0) and (n == 0).all()
    want = T.float().argmax(dim=2)[:, 0]
    assert torch.equal(out[:, 0], want.int()) and torch.equal(nxt, want.int())


def test_repeated_calls_sizes_and_graph_replay(spec, ws):
    """Calls of different sizes on one workspace, and repeats inside one CUDA graph (the scan
    launch chained to the streaming one), give the same outputs."""
    a = W.mtp_greedy("cuda", R=40, gamma=3, V=30000, seed=3)
    b = W.mtp_greedy("cuda", R=7, gamma=5, V=12000, seed=4)
    ra = [x.clone() for x in spec.spec_mtp_greedy(a.U, a.target, workspace=ws)]
    rb = [x.clone() for x in spec.spec_mtp_greedy(b.U, b.target, workspace=ws)]
    outs = [torch.empty_like(x) for x in ra]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    ws.for_op(spec.SPEC_OP_MTP_GREEDY, 40, 3, 30000, 0, stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(3):
            spec.spec_mtp_greedy(a.U, a.target, draft_tokens=outs[0], accept_len=outs[1],
                                 out_tokens=outs[2], next_anchor=outs[3], workspace=ws,
                                 stream=stream)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(ra, outs):
        assert torch.equal(x, y)
    rb2 = spec.spec_mtp_greedy(b.U, b.target, workspace=ws)
    torch.cuda.synchronize()
    for x, y in zip(rb, rb2):
        assert torch.equal(x, y)


def test_nonfinite_row_and_bad_length_are_flagged(spec):
    """A draft row of NaN sets SPEC_DEV_NONFINITE (its argmax reads 0); a length outside
    [0, gamma] sets SPEC_DEV_BAD_LENGTH and is clamped, as in spec_verify_greedy."""
    w = spec.Workspace(device="cuda")
    D = torch.randn(3, 2, 9000, dtype=torch.bfloat16)
    T = torch.randn(3, 3, 9000, dtype=torch.bfloat16)
    D[1, 0, :] = float("nan")
    got = spec.spec_mtp_greedy(D.cuda(), T.cuda(), workspace=w)
    torch.cuda.synchronize()
    assert w.status() & spec.SPEC_DEV_NONFINITE
    assert int(got[0][1, 0]) == 0
    w2 = spec.Workspace(device="cuda")
    D[1, 0, :] = 0.0
    ln = torch.tensor([-1, 5, 1], dtype=torch.int32)
    got = spec.spec_mtp_greedy(D.cuda(), T.cuda(), ln.cuda(), workspace=w2)
    ref = _two_call(spec, D.cuda(), T.cuda(), torch.tensor([0, 2, 1], dtype=torch.int32).cuda(),
                    spec.Workspace(device="cuda"))
    torch.cuda.synchronize()
    assert w2.status() & spec.SPEC_DEV_BAD_LENGTH
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
