"""Flattened (variable-length) verify batch ("[DeepSeek-6] DSpark", section 7) through the C ABI.

The packed layout is checked bit-exactly against the oracle's; the verify entry points on a
packed target are checked against the oracle's padded-layout verification with the same lengths
(the layouts hold the same rows, so the decisions are the same) and, bit-exactly, against the
library's own padded-layout entry points. Rows of the packed target past the batch hold NaN: a
kernel that read one would raise the non-finite status bit or change a result."""
import numpy as np
import pytest
import torch

import oracle
from draft_sampling_verification_markov_gb300 import workloads as W
from gpu_util import compare_proposals, compare_verify, to_dev

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


def _lengths(R, gamma, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, gamma + 1, R).astype(np.int32))


def _pack(padded, lengths):
    """Packed copy of a padded [R, gamma+1, ...] array by the oracle's layout; rows past the
    batch are NaN."""
    R, g1 = padded.shape[:2]
    offs = oracle.flat_layout(lengths, g1 - 1)["offsets"]
    out = torch.full((R * g1,) + tuple(padded.shape[2:]), float("nan"), dtype=padded.dtype)
    for r in range(R):
        l = int(lengths[r])
        out[offs[r]:offs[r] + l + 1] = padded[r, :l + 1]
    return out


@pytest.mark.parametrize("R,gamma", [(0, 3), (1, 1), (5, 3), (300, 7), (5000, 16), (2049, 0)])
def test_flat_layout_bit_exact(spec, ws, R, gamma):
    lengths = _lengths(R, gamma, R + gamma)
    offsets, row_req, row_pos = spec.spec_flat_layout(lengths.cuda(), gamma, workspace=ws)
    ref = oracle.flat_layout(lengths, gamma)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(row_req.cpu().numpy(), ref["row_req"])
    np.testing.assert_array_equal(row_pos.cpu().numpy(), ref["row_pos"])


def test_flat_layout_flags_bad_lengths(spec):
    w = spec.Workspace(device="cuda")
    lengths = torch.tensor([2, -1, 9, 0], dtype=torch.int32)
    offsets, _, _ = spec.spec_flat_layout(lengths.cuda(), 3, workspace=w, markers=False)
    ref = oracle.flat_layout(lengths.clamp(0, 3), 3)       # clamped, as the header states
    np.testing.assert_array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert w.status() == spec.SPEC_DEV_BAD_LENGTH


def test_target_stats_flat_reads_only_the_batch(spec, ws):
    wl = W.markov_rejection("cpu", R=37, gamma=5, V=4104, rank=64, seed=61, temperature=0.7)
    lengths = _lengths(37, 5, 3)
    packed = _pack(wl.target, lengths).cuda()
    offsets, _, _ = spec.spec_flat_layout(lengths.cuda(), 5, workspace=ws, markers=False)
    stats = torch.full((37 * 6, 2), 12345.0, device="cuda")
    spec.spec_target_stats_flat(packed, 0.7, offsets, 5, stats=stats, workspace=ws)
    dense = spec.spec_target_stats(wl.target.cuda(), 0.7, workspace=ws).view(37, 6, 2)
    B = int(offsets[-1].item())
    np.testing.assert_array_equal(stats[:B].cpu().numpy(), _pack(dense.cpu(), lengths)[:B].numpy())
    assert (stats[B:] == 12345.0).all()


def test_greedy_flat_bit_exact(spec, ws):
    wl = W.mtp_greedy("cpu", R=17, gamma=3, V=129280, seed=5)
    g = to_dev(wl, "cuda")
    toks, _, _ = spec.spec_markov_propose(g["U"], None, None, None, None, 0.0, workspace=ws,
                                          want_stats=False)
    lengths = torch.tensor([i % 4 for i in range(17)], dtype=torch.int32)
    offsets, _, _ = spec.spec_flat_layout(lengths.cuda(), 3, workspace=ws, markers=False)
    n, out, nxt = spec.spec_verify_greedy_flat(_pack(wl.target, lengths).cuda(), toks,
                                               lengths.cuda(), offsets, workspace=ws)
    rv = oracle.verify_greedy(wl.target, toks.cpu(), lengths)
    np.testing.assert_array_equal(n.cpu().numpy(), rv["accept_len"])
    np.testing.assert_array_equal(out.cpu().numpy(), rv["out_tokens"])
    np.testing.assert_array_equal(nxt.cpu().numpy(), rv["next_anchor"])


FLAT_CASES = [
    # R, gamma, V, rank, wdtype
    (130, 3, 1000, 256, "bf16"),     # tensor-core residual pass, two 128-row tiles
    (9, 4, 4104, 64, "bf16"),
    (6, 3, 777, 32, "bf16"),         # CUDA-core producer
    (7, 3, 1000, 48, "f32"),
    (5, 4, 2048, 0, "bf16"),         # no Markov head: streaming residual
]


@pytest.mark.parametrize("R,gamma,V,rank,wdt", FLAT_CASES)
@pytest.mark.parametrize("precomputed_stats", [False, True])
def test_rejection_flat_matches_padded_and_oracle(spec, ws, R, gamma, V, rank, wdt,
                                                   precomputed_stats):
    wl = W.markov_rejection("cpu", R=R, gamma=gamma, V=V, rank=max(rank, 1), seed=300 + V,
                            temperature=0.8)
    if rank == 0:
        wl.W1 = wl.W2 = None
    elif wdt == "f32":
        wl.W1, wl.W2 = wl.W1.float(), wl.W2.float()
        wl.U, wl.target = wl.U.float(), wl.target.float()
    g = to_dev(wl, "cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g.get("W1"), g.get("W2"), g["anchors"],
                                                 g["u_draft"], 0.8, rank=rank, workspace=ws)
    lengths = _lengths(R, gamma, V)
    ld = lengths.cuda()
    offsets, _, _ = spec.spec_flat_layout(ld, gamma, workspace=ws, markers=False)
    packed = _pack(wl.target, lengths).cuda()
    tstats = (spec.spec_target_stats_flat(packed, 0.8, offsets, gamma, workspace=ws)
              if precomputed_stats else None)
    args = (g["U"], g.get("W1"), g.get("W2"), g["anchors"], toks, logp, stats, g["u_accept"],
            g["u_resid"], 0.8)
    n, out, nxt = spec.spec_verify_rejection_flat(packed, *args, ld, offsets, rank=rank,
                                                  target_stats=tstats, workspace=ws)
    dn, dout, dnxt = spec.spec_verify_rejection(g["target"], *args, ld, rank=rank, workspace=ws)
    # the same rows through the same kernels: identical decisions and draws
    assert torch.equal(n, dn) and torch.equal(out, dout) and torch.equal(nxt, dnxt)
    ref = oracle.markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, 0.8, rank=rank)
    same = compare_proposals(toks, logp, stats, ref)
    rv = oracle.verify_rejection(wl.target, wl.U, wl.W1, wl.W2, wl.anchors, toks.cpu(),
                                 wl.u_accept, wl.u_resid, 0.8, lengths, rank=rank)
    gn, go, gx = n.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy()
    compare_verify(gn, go, gx, rv)
    assert (gn <= lengths.numpy()).all()
    assert same.any()


def test_masked_rejection_flat(spec, ws):
    R, gamma, V, rank = 40, 4, 2048, 64
    wl = W.markov_rejection("cpu", R=R, gamma=gamma, V=V, rank=rank, seed=71, temperature=1.0)
    allowed = torch.from_numpy(np.random.default_rng(4).integers(
        0, 1 << 32, (R, V // 32), dtype=np.uint64).astype(np.uint32).view(np.int32))
    g = to_dev(wl, "cuda")
    al = allowed.cuda()
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"],
                                                 g["u_draft"], 1.0, workspace=ws, allowed=al)
    lengths = _lengths(R, gamma, 9)
    ld = lengths.cuda()
    offsets, _, _ = spec.spec_flat_layout(ld, gamma, workspace=ws, markers=False)
    args = (g["U"], g["W1"], g["W2"], g["anchors"], toks, logp, stats, g["u_accept"],
            g["u_resid"], 1.0)
    n, out, nxt = spec.spec_verify_rejection_flat(_pack(wl.target, lengths).cuda(), *args, ld,
                                                  offsets, workspace=ws, allowed=al)
    dn, dout, dnxt = spec.spec_verify_rejection(g["target"], *args, ld, workspace=ws, allowed=al)
    assert torch.equal(n, dn) and torch.equal(out, dout) and torch.equal(nxt, dnxt)


def test_scheduler_to_flat_verify(spec, ws):
    """Scheduler lengths -> packed batch of exactly B rows -> verify, as one device-resident
    chain; equal to the padded-layout verify with the same lengths."""
    wl = W.full_loop("cpu", R=64, gamma=5, V=2048, rank=64, iterations=1, seed=90)
    g = to_dev(wl, "cuda")
    toks, logp, stats = spec.spec_markov_propose(g["U"], g["W1"], g["W2"], g["anchors"],
                                                 g["u_draft"][0], wl.temperature, workspace=ws)
    _, surv = spec.spec_tv_confidence(g["U"], g["target"], g["W1"], g["W2"], g["anchors"], toks,
                                      wl.temperature, draft_stats=stats, workspace=ws)
    lengths, B, _ = spec.spec_schedule_prefix(surv, g["sps"], workspace=ws)
    offsets, row_req, row_pos = spec.spec_flat_layout(lengths, 5, workspace=ws)
    assert int(offsets[-1].item()) == int(B.item())
    lc = lengths.cpu()
    ref = oracle.flat_layout(lc, 5)
    np.testing.assert_array_equal(row_req.cpu().numpy(), ref["row_req"])
    np.testing.assert_array_equal(row_pos.cpu().numpy(), ref["row_pos"])
    args = (g["U"], g["W1"], g["W2"], g["anchors"], toks, logp, stats, g["u_accept"][0],
            g["u_resid"][0], wl.temperature)
    n, out, nxt = spec.spec_verify_rejection_flat(_pack(wl.target, lc).cuda(), *args, lengths,
                                                  offsets, workspace=ws)
    dn, dout, dnxt = spec.spec_verify_rejection(g["target"], *args, lengths, workspace=ws)
    assert torch.equal(n, dn) and torch.equal(out, dout) and torch.equal(nxt, dnxt)


@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 1000), (torch.float32, 2), (torch.float32, 7)])
def test_flat_pack_copies_only_the_scheduled_rows(spec, ws, dtype, width):
    """spec_flat_pack: padded row (r, i <= l_r) lands on packed row offsets[r] + i; rows past
    B keep what they held (NaN here), whatever the row width (16-byte or 4-byte copies)."""
    R, gamma = 37, 5
    g = torch.Generator().manual_seed(width)
    src = torch.randn(R, gamma + 1, width, generator=g).to(dtype).cuda()
    lengths = torch.randint(0, gamma + 1, (R,), generator=g, dtype=torch.int32).cuda()
    offsets, _, _ = spec.spec_flat_layout(lengths, gamma, markers=False, workspace=ws)
    out = torch.full((R * (gamma + 1), width), float("nan"), dtype=dtype, device="cuda")
    spec.spec_flat_pack(src, lengths, offsets, out=out, workspace=ws)
    torch.cuda.synchronize()
    ln = lengths.cpu().tolist()
    want = torch.cat([src[r, :ln[r] + 1] for r in range(R)])
    B = want.shape[0]
    assert int(offsets[-1]) == B
    assert torch.equal(out[:B], want)
    assert torch.isnan(out[B:].float()).all()
