"""Shared helpers of the GPU parity tests (comparison rules against the oracle)."""
import numpy as np
import torch

# Tolerances. Token ids, accept lengths and scheduler outputs are compared exactly. A sampled
# token may differ only where the oracle's CDF margin is below MARGIN (the GPU accumulates in
# fp32); such cases are counted and reported. Probabilities: relative 1e-5, i.e. 1e-5 absolute
# on log-probabilities and log-normalisers; confidences 1e-5 relative with a 1e-7 absolute floor.
MARGIN = 1e-6
LOG_TOL = 1e-5
CONF_RTOL, CONF_ATOL = 1e-5, 1e-7


# Session totals of every comparison with the oracle (printed in the test summary, see
# conftest.py): requests compared, requests identical to the oracle, and the mismatches the
# margin rule allowed (sampled draft tokens whose oracle CDF margin is below MARGIN; acceptance
# decisions within MARGIN of the ratio or final draws below MARGIN, on the verify side).
PARITY = {"proposal_requests": 0, "proposal_exact": 0, "proposal_margin_cases": 0,
          "verify_requests": 0, "verify_exact": 0, "verify_margin_cases": 0}


def to_dev(wl, dev):
    return {k: v.to(dev) for k, v in wl.tensors().items()}


def compare_proposals(gpu_tokens, gpu_logp, gpu_stats, ref, greedy=False, report=None):
    """Compare GPU proposals with the oracle's. Returns the boolean mask of requests whose
    proposals are identical. Where a request first differs, the oracle's decision margin must be
    below MARGIN (sampling) -- greedy proposals must be identical everywhere."""
    gt = gpu_tokens.cpu().numpy()
    rt = ref["tokens"]
    same = (gt == rt).all(axis=1)
    if greedy:
        bad = np.nonzero(~same)[0]
        assert len(bad) == 0, f"greedy proposals differ for requests {bad[:10]}"
    n_margin = 0
    for r in np.nonzero(~same)[0]:
        k = int(np.argmax(gt[r] != rt[r]))
        assert ref["margin"][r, k] < MARGIN, (
            f"request {r} position {k + 1}: token {gt[r, k]} vs oracle {rt[r, k]} with margin "
            f"{ref['margin'][r, k]:.3e}")
        n_margin += 1
    # probabilities on the common prefix of every request
    if gpu_logp is not None:
        gl = gpu_logp.cpu().numpy().astype(np.float64)
        gs = gpu_stats.cpu().numpy().astype(np.float64)
        agree = np.cumprod(gt == rt, axis=1).astype(bool)
        # position k's distribution depends only on tokens before k
        cond = np.concatenate([np.ones((gt.shape[0], 1), bool), agree[:, :-1]], axis=1)
        dl = np.abs(gl - ref["logp"])[agree]
        assert dl.size == 0 or dl.max() <= LOG_TOL, f"log p_d differs by {dl.max():.3e}"
        ln_g = gs[..., 0] + gs[..., 1]
        ln_r = ref["stats"][..., 0] + ref["stats"][..., 1]
        dn = (np.abs(ln_g - ln_r) / np.maximum(1.0, np.abs(ln_r)))[cond]
        assert dn.size == 0 or dn.max() <= LOG_TOL, f"log-normaliser differs by {dn.max():.3e}"
    if report is not None:
        report["margin_mismatches"] = report.get("margin_mismatches", 0) + n_margin
    PARITY["proposal_requests"] += int(same.size)
    PARITY["proposal_exact"] += int(same.sum())
    PARITY["proposal_margin_cases"] += n_margin
    return same


def compare_verify(accept_len, out_tokens, next_anchor, rv, same=None, report=None):
    """Compare rejection-verification outputs with the oracle's, request by request. A request
    whose proposals differ from the oracle's (`same` False) is not compared; the others must
    agree exactly unless the oracle's acceptance ratio or final draw lies within MARGIN of the
    uniform (counted). Returns the number of requests compared."""
    gn, go = np.asarray(accept_len), np.asarray(out_tokens)
    gx = None if next_anchor is None else np.asarray(next_anchor)
    R = gn.shape[0]
    same = np.ones(R, bool) if same is None else np.asarray(same)
    amb = (np.nan_to_num(rv["accept_margin"], nan=1.0) < MARGIN).any(axis=1)
    amb |= rv["resid_margin"] < MARGIN
    diff = (gn != rv["accept_len"]) | (go != rv["out_tokens"]).any(axis=1)
    if gx is not None:
        diff |= gx != rv["next_anchor"]
    bad = same & diff & ~amb
    assert not bad.any(), f"verify differs for requests {np.nonzero(bad)[0][:10]}"
    n_margin = int((same & diff & amb).sum())
    if report is not None:
        report["verify_margin_cases"] = report.get("verify_margin_cases", 0) + n_margin
    PARITY["verify_requests"] += int(same.sum())
    PARITY["verify_exact"] += int((same & ~diff).sum())
    PARITY["verify_margin_cases"] += n_margin
    return int(same.sum())


def assert_conf_close(gpu, ref, what="confidence"):
    g = gpu.cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    tol = CONF_RTOL * np.abs(ref) + CONF_ATOL
    assert np.all(err <= tol), f"{what}: max excess {np.max(err - tol):.3e}"


def bf16(t):
    return t.to(torch.bfloat16)
