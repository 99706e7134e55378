#!/usr/bin/env python
"""Benchmark of the speculative-decoding hot path on GB300.

Workload (N=1): DSpark Markov sampling + lossless rejection verification, R=256 requests,
gamma=7 proposed positions, V=129280, Markov rank 256, bf16 logits and weights, T=1.
One step = the whole hot path over one batch: gamma serial Markov proposal positions
(tensor-core bias GEMM fused with softmax partials, then inverse-CDF sampling) in one
persistent launch that also streams the target rows into their softmax normalisers, the
acceptance scan, and the residual / bonus draw.

Metric: draft + verify logit rows per second, rows = R*gamma + R*(gamma+1) = 3840 per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, fp64) on a bounded sample of the same workload.
For N > 1 (torchrun, one rank per GPU) every rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft+verify logit rows/s at V=129280, R=256 (HBM GB/s, % of peak)"
UNIT = "rows/s"
WORKLOAD = dict(R=256, gamma=7, V=129280, rank=256, temperature=1.0, seed=1003)
# timed regions of K steps each; `value` is their median
REPEATS = 5
# the step's proposal and target normalisers in one call (spec_markov_propose_target_stats):
# 0.383 ms against 0.401 ms per step as two calls, on one box
FUSED = True


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-other-configs", action="store_true")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_seed(base, rank):
    """Each replica (one rank per GPU) draws its own workload of the same shape."""
    return base + 100 * rank


def max_over_ranks(x, dist=None, device="cpu"):
    """The maximum of a per-rank time over all ranks (the timing rule for N > 1)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step, steps, world, ms):
    """Units of all ranks per second of the slowest rank."""
    return units_per_step * steps * world / (ms / 1e3)


def config_dict(extra=None):
    c = {"workload": "markov_rejection: Markov-head sampling + rejection verify, R=256 gamma=7 "
                     "V=129280 rank=256 bf16 T=1",
         "R": WORKLOAD["R"], "gamma": WORKLOAD["gamma"], "V": WORKLOAD["V"],
         "rank": WORKLOAD["rank"], "temperature": WORKLOAD["temperature"],
         "storage_dtype": "bf16",
         "rows_per_step": WORKLOAD["R"] * (2 * WORKLOAD["gamma"] + 1),
         "l2": "inputs larger than L2 (1.06 GB of logits per step vs 129 MB L2)"}
    if extra:
        c.update(extra)
    return c


def algorithmic_bytes_per_step():
    """What one step must touch: U and the target read once, W2 read once, W1 row gathers."""
    R, g, V, r = (WORKLOAD[k] for k in ("R", "gamma", "V", "rank"))
    return 2 * (R * g * V + R * (g + 1) * V + V * r + R * g * r)


def class_bytes_per_launch():
    """Algorithmic bytes of one launch of each kernel class in the step (bf16 everywhere):
    the persistent proposal reads U, W2 and the gathered W1 rows (and, in the fused entry point,
    the target); the residual pass reads each request's final U and target rows, W2 and W1 rows;
    the target normalisers read the target; selects and scans read only partials."""
    R, g, V, r = (WORKLOAD[k] for k in ("R", "gamma", "V", "rank"))
    propose = 2 * (R * g * V + V * r + R * g * r) + (2 * R * (g + 1) * V if FUSED else 0)
    return {4: propose, 0: 2 * (2 * R * V + V * r + R * r), 1: 2 * R * (g + 1) * V,
            2: 8 * R * ((V + 63) // 64), 3: 0}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 6:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        win = [p for t, p in self.samples if t0 - 0.05 <= t <= t1 + 0.05]
        if not win and self.samples:
            mid = (t0 + t1) / 2
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[2 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win)}


# ----------------------------------------------------------------------------- profile traffic

def recorded_traffic(kernel_class):
    """DRAM bytes per launch of the dominant kernel class from the committed ncu summary
    (profiles/traffic.json), or None if absent or taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(kernel_class)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    blob = b""
    for src in rec.get("sources", []):
        f = os.path.join(ROOT, src)
        if not os.path.exists(f):
            return None
        blob += open(f, "rb").read()
    if hashlib.sha256(blob).hexdigest()[:16] != rec.get("sources_sha256_16"):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- CPU baseline

def cpu_baseline_run(wl_host, n_req):
    """Time the oracle (propose + rejection verify) on the first n_req requests. Returns
    (rows/s, seconds, proposal, verification) with the oracle's outputs."""
    import oracle
    sl = lambda t: None if t is None else t[:n_req]
    t0 = time.perf_counter()
    ref = oracle.markov_propose(sl(wl_host["U"]), wl_host["W1"], wl_host["W2"],
                                sl(wl_host["anchors"]), sl(wl_host["u_draft"]),
                                WORKLOAD["temperature"])
    rv = oracle.verify_rejection(sl(wl_host["target"]), sl(wl_host["U"]), wl_host["W1"],
                                 wl_host["W2"], sl(wl_host["anchors"]), ref["tokens"],
                                 sl(wl_host["u_accept"]), sl(wl_host["u_resid"]),
                                 WORKLOAD["temperature"])
    dt = time.perf_counter() - t0
    rows = n_req * (2 * WORKLOAD["gamma"] + 1)
    return rows / dt, dt, ref, rv


def parity_summary(ref, rv, toks, n_acc, out, margin=1e-6):
    """The GPU step's outputs against the oracle's on the same requests (the tests' rule): a
    request's proposals must be identical unless, where they first differ, the oracle's CDF
    margin is below `margin`; the verification of a request with identical proposals must be
    identical unless an acceptance ratio or the final draw lies within `margin` of its uniform.
    Mismatches outside these margins are counted, not hidden."""
    import numpy as np
    rt = ref["tokens"]
    same = (toks == rt).all(axis=1)
    margin_cases = 0
    outside = 0
    for r in np.nonzero(~same)[0]:
        k = int(np.argmax(toks[r] != rt[r]))
        if ref["margin"][r, k] < margin:
            margin_cases += 1
        else:
            outside += 1
    amb = (np.nan_to_num(rv["accept_margin"], nan=1.0) < margin).any(axis=1)
    amb |= rv["resid_margin"] < margin
    diff = (n_acc != rv["accept_len"]) | (out != rv["out_tokens"]).any(axis=1)
    return {"requests_compared": int(len(rt)), "proposals_exact": int(same.sum()),
            "margin_cases": margin_cases, "verify_exact": int((same & ~diff).sum()),
            "verify_margin_cases": int((same & diff & amb).sum()),
            "mismatches_outside_margin": outside + int((same & diff & ~amb).sum()),
            "margin": margin,
            "rule": "tokens, accept lengths and emitted tokens identical to the fp64 oracle except "
                    "at a CDF or acceptance margin below 1e-6"}


def host_sample(n_req, device):
    """The first n_req requests of the workload, drawn on `device`, copied to host."""
    from draft_sampling_verification_markov_gb300 import workloads
    wl = workloads.markov_rejection(device, R=WORKLOAD["R"], gamma=WORKLOAD["gamma"],
                                    V=WORKLOAD["V"], rank=WORKLOAD["rank"], seed=WORKLOAD["seed"],
                                    temperature=WORKLOAD["temperature"])
    out = {}
    for k, v in wl.tensors().items():
        out[k] = v[:n_req].cpu() if k not in ("W1", "W2") else v.cpu()
    del wl
    return out


def run_reference(args):
    """--impl reference: the CPU oracle, timed on the host cores, on a bounded sample."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    n_req = max(1, min(WORKLOAD["R"], threads))
    wl = host_sample(n_req, "cpu")
    for _ in range(args.warmup):
        cpu_baseline_run(wl, n_req)[:2]
    times = []
    for _ in range(args.steps):
        times.append(cpu_baseline_run(wl, n_req)[1])
    total = sum(times)
    rows = n_req * (2 * WORKLOAD["gamma"] + 1) * args.steps
    value = rows / total
    sample = (f"{n_req} of {WORKLOAD['R']} requests per step (all {WORKLOAD['gamma']} positions, "
              f"full V), CPU-drawn inputs of the same shapes and distributions")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": config_dict({"sample_requests_per_step": n_req}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, n_req),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

# ----------------------------------------------------------------------------- other configs

def graph_ms(run, stream, reps=5, warm=2, flush=None):
    """Milliseconds per replay of `run` captured as one CUDA graph on `stream`. With `flush` (a
    device buffer larger than L2) each replay is timed alone after the buffer is rewritten,
    outside the timed events, and the median is returned."""
    import torch
    stream.wait_stream(torch.cuda.current_stream())  # inputs drawn on the current stream
    with torch.cuda.stream(stream):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run()
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    stream.synchronize()
    if flush is not None:
        times = []
        for i in range(max(reps, 9)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush.fill_(i & 0xff)
                a.record(stream)
                g.replay()
                b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        return statistics.median(times)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def other_configs(spec, workloads, dev, peak):
    """The other rows of the path on their own workloads, each step one CUDA graph with inputs
    resident: the fp32 greedy toy, MTP-1 greedy verify, confidence + scheduling, and one
    iteration of the 20-iteration loop. Bytes are the algorithmic bytes the step must touch."""
    import torch
    from draft_sampling_verification_markov_gb300.loop import SpecLoop
    out = {}
    stream = torch.cuda.Stream(device=dev)
    # the toy and MTP-1 inputs fit in L2 (129 MB): their replays are timed one by one, each
    # after a 256 MB buffer is rewritten
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flushed = {"l2": "inputs smaller than L2: each replay timed alone after a 256 MB write"}

    def entry(name, ms, rows, nbytes, extra=None):
        e = {"ms_per_step": ms, "rows_per_s": rows / (ms / 1e3), "rows_per_step": rows,
             "algorithmic_bytes": nbytes, "hbm_gbs": nbytes / (ms / 1e3) / 1e9,
             "hbm_frac": nbytes / (ms / 1e3) / 1e9 / peak}
        e.update(extra or {})
        out[name] = e

    # fp32 greedy toy: Markov argmax (CUDA-core canonical chain) + greedy verify; latency-bound
    wl = workloads.greedy_toy("cuda")
    ws = spec.Workspace(device=dev)
    R, g, V = wl.R, wl.gamma, wl.V
    toks = torch.empty(R, g, dtype=torch.int32, device=dev)
    res = [torch.empty(R, dtype=torch.int32, device=dev),
           torch.empty(R, g + 1, dtype=torch.int32, device=dev),
           torch.empty(R, dtype=torch.int32, device=dev)]
    for op in range(6):
        ws.for_op(op, R, g, V, wl.rank, stream)

    def toy():
        spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, None, 0.0, draft_tokens=toks,
                                 want_stats=False, workspace=ws, stream=stream)
        spec.spec_verify_greedy(wl.target, toks, accept_len=res[0], out_tokens=res[1],
                                next_anchor=res[2], workspace=ws, stream=stream)
    ms = graph_ms(toy, stream, flush=flush)
    nbytes = (wl.U.numel() + wl.target.numel() + wl.W2.numel()) * 4
    entry("greedy_toy_fp32_R4_g4_V32000", ms, R * (2 * g + 1), nbytes,
          {"bound": "latency", "us_per_step": ms * 1e3, **flushed})
    del wl

    # MTP-1 greedy: rank-0 argmax proposal + greedy verify. One batch (116 MB) fits in L2, so
    # the timed graph runs three batches of the same shape in turn (348 MB): each step reads
    # inputs that two other steps have pushed out of L2 since it last ran
    wls = [workloads.mtp_greedy("cuda", seed=1002 + 100 * i) for i in range(3)]
    wl = wls[0]
    R, g, V = wl.R, wl.gamma, wl.V
    toks = torch.empty(R, g, dtype=torch.int32, device=dev)
    res = [torch.empty(R, dtype=torch.int32, device=dev),
           torch.empty(R, g + 1, dtype=torch.int32, device=dev),
           torch.empty(R, dtype=torch.int32, device=dev)]
    for op in range(7):
        ws.for_op(op, R, g, V, 0, stream)

    def mtp():
        for w in wls:
            spec.spec_mtp_greedy(w.U, w.target, draft_tokens=toks, accept_len=res[0],
                                 out_tokens=res[1], next_anchor=res[2], workspace=ws,
                                 stream=stream)
    ms = graph_ms(mtp, stream) / len(wls)
    ms_alone = graph_ms(mtp, stream, flush=flush) / len(wls)
    entry("mtp_greedy_R64_g3_V129280", ms, R * (2 * g + 1),
          (wl.U.numel() + wl.target.numel()) * 2,
          {"mean_accept_len": float(res[0].float().mean()),
           "l2": "three batches in turn (348 MB) per replay, replays back to back",
           "ms_per_step_l2_flushed_replays": ms_alone})
    del wl, wls, flush

    # confidence + scheduling: proposal, target normalisers, TV labels + survival, scheduler
    wl = workloads.confidence_scheduling("cuda")
    R, g, V = wl.R, wl.gamma, wl.V
    toks = torch.empty(R, g, dtype=torch.int32, device=dev)
    logp = torch.empty(R, g, dtype=torch.float32, device=dev)
    dst = torch.empty(R, g, 2, dtype=torch.float32, device=dev)
    tst = torch.empty(R * (g + 1), 2, dtype=torch.float32, device=dev)
    conf = torch.empty(R, g, dtype=torch.float32, device=dev)
    surv = torch.empty(R, g, dtype=torch.float32, device=dev)
    lens = torch.empty(R, dtype=torch.int32, device=dev)
    B = torch.empty(1, dtype=torch.int32, device=dev)
    th = torch.empty(1, dtype=torch.float64, device=dev)
    sps = wl.sps.to(dev)
    for op in range(6):
        ws.for_op(op, R, g, V, wl.rank, stream)

    def conf_sched():
        spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, wl.temperature,
                                 draft_tokens=toks, draft_logp=logp, draft_stats=dst,
                                 workspace=ws, stream=stream)
        spec.spec_target_stats(wl.target, wl.temperature, stats=tst, workspace=ws,
                               stream=stream)
        spec.spec_tv_confidence(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, toks,
                                wl.temperature, draft_stats=dst, target_stats=tst, conf=conf,
                                survival=surv, workspace=ws, stream=stream)
        spec.spec_schedule_prefix(surv, sps, lengths=lens, B_out=B, theta_out=th,
                                  workspace=ws, stream=stream)
    ms = graph_ms(conf_sched, stream, reps=3)
    entry("confidence_scheduling_R512_g16_V129280", ms, R * (2 * g + 1),
          (wl.U.numel() + wl.target.numel() + wl.W2.numel()) * 2,
          {"scheduled_B": int(B.item()), "note": "U and target counted once; the TV pass "
           "reads them a second time"})
    del wl, toks, logp, dst, tst, conf, surv

    # the 20-iteration loop: two chained iterations per graph, time per iteration
    wl = workloads.full_loop("cuda", iterations=2)
    lp = SpecLoop(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, wl.u_draft, wl.u_accept,
                  wl.u_resid, wl.temperature, wl.sps.to(dev), iterations=2)
    ms = graph_ms(lambda: lp.run(), stream, reps=3) / 2
    R, g = wl.R, wl.gamma
    entry("full_loop_R1024_g16_V129280_per_iteration", ms, R * (2 * g + 1),
          (wl.U.numel() + wl.target.numel() + wl.W2.numel()) * 2,
          {"mean_emitted_per_request": float(lp.emitted_tokens().float().mean())})
    assert ws.status() == 0 and lp.ws.status() == 0, "device status word set"
    padded_out = lp.out_tokens.clone()
    del lp
    torch.cuda.empty_cache()

    # the same iterations verifying the flattened batch (packed rows, per-request offsets); the
    # packing copy of the B scheduled rows stands in for a target model that writes only them
    lp = SpecLoop(wl.U, wl.target, wl.W1, wl.W2, wl.anchors, wl.u_draft, wl.u_accept,
                  wl.u_resid, wl.temperature, wl.sps.to(dev), iterations=2, flat=True)
    ms_flat = graph_ms(lambda: lp.run(), stream, reps=3) / 2
    B = float(lp.batch.float().mean())
    row_bytes = wl.V * wl.target.element_size()
    entry("full_loop_flat_R1024_g16_V129280_per_iteration", ms_flat, R * (2 * g + 1),
          (wl.U.numel() + wl.target.numel() + wl.W2.numel()) * 2,
          {"scheduled_B": B, "padded_rows": R * (g + 1),
           "packed_bytes_per_iteration": 2 * B * row_bytes,
           "padded_ms_per_iteration": ms,
           "same_outputs_as_padded": bool(torch.equal(padded_out, lp.out_tokens)),
           "note": "packing copies only the B scheduled target rows (read + write); "
                   "verification then reads the packed rows"})
    assert lp.ws.status() == 0, "device status word set"
    del wl, lp
    torch.cuda.empty_cache()
    return out


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec, workloads

    W = WORKLOAD
    wl = workloads.markov_rejection("cuda", R=W["R"], gamma=W["gamma"], V=W["V"], rank=W["rank"],
                                    seed=replica_seed(W["seed"], rank),
                                    temperature=W["temperature"])
    R, g, V = W["R"], W["gamma"], W["V"]
    T = W["temperature"]
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # the inputs are drawn on that stream
    ws = spec.Workspace(device=dev)
    for op in range(6):
        ws.for_op(op, R, g, V, W["rank"], stream)
    toks = torch.empty(R, g, dtype=torch.int32, device=dev)
    logp = torch.empty(R, g, dtype=torch.float32, device=dev)
    dstats = torch.empty(R, g, 2, dtype=torch.float32, device=dev)
    tstats = torch.empty(R * (g + 1), 2, dtype=torch.float32, device=dev)
    n_acc = torch.empty(R, dtype=torch.int32, device=dev)
    out = torch.empty(R, g + 1, dtype=torch.int32, device=dev)
    nxt = torch.empty(R, dtype=torch.int32, device=dev)

    def step(U, target, anchors, u_draft, u_acc, u_res):
        if FUSED:
            spec.spec_markov_propose_target_stats(U, wl.W1, wl.W2, anchors, u_draft, T, target,
                                                  draft_tokens=toks, draft_logp=logp,
                                                  draft_stats=dstats, target_stats=tstats,
                                                  workspace=ws, stream=stream)
        else:
            spec.spec_markov_propose(U, wl.W1, wl.W2, anchors, u_draft, T, draft_tokens=toks,
                                     draft_logp=logp, draft_stats=dstats, workspace=ws,
                                     stream=stream)
            spec.spec_target_stats(target, T, stats=tstats, workspace=ws, stream=stream)
        spec.spec_verify_rejection(target, U, wl.W1, wl.W2, anchors, toks, logp, dstats, u_acc,
                                   u_res, T, target_stats=tstats, accept_len=n_acc,
                                   out_tokens=out, next_anchor=nxt, workspace=ws, stream=stream)

    inputs = (wl.U, wl.target, wl.anchors, wl.u_draft, wl.u_accept, wl.u_resid)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(*inputs)
    torch.cuda.synchronize()
    assert ws.status() == 0, "device status word set during warm-up"

    # the step as one CUDA graph (the library's calls neither synchronise nor allocate)
    launches0 = spec.lib().spec_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(*inputs)
    launches_per_step = spec.lib().spec_launch_count() - launches0
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            graph.replay()
    torch.cuda.synchronize()

    # timed regions: REPEATS times K replays of the step, no per-launch instrumentation; each
    # region is bracketed by a barrier and a synchronisation and timed with CUDA events on the
    # launch stream; `value` is the median region, its spread reported beside it
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    region_ms = []
    w0 = time.time()
    for _ in range(REPEATS):
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        region_ms.append(max_over_ranks(t_start.elapsed_time(t_end), pg, dev))
    w1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    launches = launches_per_step * args.steps
    ms = sorted(region_ms)[len(region_ms) // 2]
    assert ws.status() == 0, "device status word set during the timed region"
    # the step's outputs (every replay computes the same ones), for the parity check below
    gpu_out = {"tokens": toks.cpu().numpy(), "accept_len": n_acc.cpu().numpy(),
               "out_tokens": out.cpu().numpy()}
    rows_per_step = R * (2 * g + 1)
    value = whole_job_rate(rows_per_step, args.steps, world, ms)
    spread = {"regions": REPEATS, "steps_per_region": args.steps,
              "value_min": whole_job_rate(rows_per_step, args.steps, world, max(region_ms)),
              "value_max": whole_job_rate(rows_per_step, args.steps, world, min(region_ms)),
              "ms_per_step_regions": [x / args.steps for x in region_ms]}

    # per-class launch durations, live: the same step captured with caller-owned CUDA events
    # around every library launch (on the launch stream), replayed and read back replay by
    # replay. The events cost about 15 % of a step, so they stay out of the region above.
    import ctypes
    caps = {kc: g + 2 for kc in range(5)}   # at most this many launches per step and class
    ev, keep = {}, []
    for kc, cap in caps.items():
        b = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
        for x in b + e:
            x.record(stream)                      # materialise the CUDA event handles
        ev[kc] = (b, e)
    torch.cuda.synchronize()
    for kc, (b, e) in ev.items():
        bh = (ctypes.c_void_p * caps[kc])(*[x.cuda_event for x in b])
        eh = (ctypes.c_void_p * caps[kc])(*[x.cuda_event for x in e])
        keep.append((bh, eh))
        assert spec.lib().spec_trace_events(kc, bh, eh, caps[kc]) == 0
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        step(*inputs)
    counts = {kc: spec.lib().spec_trace_count(kc) for kc in range(5)}
    for kc in range(5):
        spec.lib().spec_trace_events(kc, None, None, 0)
    n_prof = max(1, min(args.steps, 50))
    totals = {kc: [0.0, 0] for kc in range(5)}
    for _ in range(n_prof):
        with torch.cuda.stream(stream):
            graph_ev.replay()
        stream.synchronize()
        for kc in range(5):
            b, e = ev[kc]
            for i in range(counts[kc]):
                totals[kc][0] += b[i].elapsed_time(e[i])
                totals[kc][1] += 1
    # scaled to the K timed steps: (total ms, launches)
    totals = {kc: (v[0] * args.steps / n_prof, v[1] * args.steps / n_prof)
              for kc, v in totals.items()}
    dom = max(totals, key=lambda k: totals[k][0])
    names = {0: "markov_producer", 1: "stream_rows", 2: "select", 3: "other",
             4: "persistent_proposal"}
    bytes_per_launch = class_bytes_per_launch()
    dur_s = totals[dom][0] / max(totals[dom][1], 1) / 1e3
    achieved = bytes_per_launch[dom] / dur_s / 1e9
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        peak, peak_src = 6800.0, "fallback"
    traffic = recorded_traffic(names[dom])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": names[dom],
                "peak_source": peak_src,
                "launch_ms": 1e3 * dur_s,
                "step_hbm_frac": algorithmic_bytes_per_step() * args.steps / (ms / 1e3) / 1e9 / peak,
                "step_hbm_frac_of_8tbs_nominal":
                    algorithmic_bytes_per_step() * args.steps / (ms / 1e3) / 1e9 / 8000.0,
                "class_ms_per_step": {names[k]: totals[k][0] / args.steps for k in totals},
                "algorithmic_bytes_per_launch": bytes_per_launch[dom],
                "class_launches_per_step": {names[k]: totals[k][1] / args.steps
                                            for k in totals}}
    # the W2 projection on the tensor pipe: 2 * R * rank * V flops per position (gamma in the
    # persistent proposal, one in the residual pass), against the bf16 dense peak
    mk = (totals[0][0] + totals[4][0], totals[0][1] + totals[4][1] * g)
    if mk[1] > 0:
        flops = 2.0 * R * W["rank"] * V * mk[1]
        # timed inside a long step: the sustained figure
        bf16 = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
        tf = flops / (mk[0] / 1e3) / 1e12
        roofline["w2_projection"] = {"bound": "tensor", "achieved": tf, "peak": bf16,
                                     "unit": "TFLOP/s", "frac": tf / bf16,
                                     "note": "flops over the tensor-core launches' time (the "
                                             "persistent proposal and the residual pass); "
                                             "they are not tensor-bound"}

    # end to end through the C ABI from pinned host buffers (weights stay resident): every step
    # copies its inputs host -> device and reads its outputs back. Two device input buffers let
    # the copy of step i+1 (copy stream) overlap the compute of step i (launch stream).
    e2e = None
    if args.e2e_steps > 0:
        host = [x.cpu().pin_memory() for x in inputs]
        dbuf = [[torch.empty_like(x) for x in inputs] for _ in range(2)]
        h_out = [torch.empty(R, g + 1, dtype=torch.int32).pin_memory() for _ in range(2)]
        h_n = [torch.empty(R, dtype=torch.int32).pin_memory() for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in host)
        d2h = h_out[0].numel() * 4 + h_n[0].numel() * 4
        cstream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]

        def copy_in(i):
            b = i % 2
            with torch.cuda.stream(cstream):
                cstream.wait_event(consumed[b])          # the buffer's previous step is done
                for dd, hh in zip(dbuf[b], host):
                    dd.copy_(hh, non_blocking=True)
                copied[b].record(cstream)

        def compute(i):
            b = i % 2
            with torch.cuda.stream(stream):
                stream.wait_event(copied[b])
                step(*dbuf[b])
                consumed[b].record(stream)
                h_out[b].copy_(out, non_blocking=True)
                h_n[b].copy_(n_acc, non_blocking=True)

        def run_e2e(k):
            copy_in(0)
            for i in range(k):
                if i + 1 < k:
                    copy_in(i + 1)
                compute(i)

        for b in range(2):
            consumed[b].record(stream)
        run_e2e(2)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run_e2e(args.e2e_steps)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(1e3 * (time.perf_counter() - t0), pg, dev)
        e2e = {"value": whole_job_rate(rows_per_step, args.e2e_steps, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.e2e_steps,
               "note": "inputs copied from pinned host memory every step (about 210 GB/s on "
                       "this host link), overlapped with the previous step's compute"}

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.num_threads()
        # a bounded sample: all requests of one step, repeated until about 10 s of CPU time
        n_req = R
        wl_h = {k: (v[:n_req].cpu() if k not in ("W1", "W2") else v.cpu())
                for k, v in wl.tensors().items()}
        dt, reps = 0.0, 0
        while reps < 4 and (reps == 0 or dt < 10.0):
            _, t_run, ref_p, ref_v = cpu_baseline_run(wl_h, n_req)
            dt += t_run
            reps += 1
        parity = parity_summary(ref_p, ref_v, gpu_out["tokens"], gpu_out["accept_len"],
                                gpu_out["out_tokens"])
        v_cpu = reps * n_req * (2 * g + 1) / dt
        cpu = {"value": v_cpu, "unit": UNIT, "cores": min(threads, n_req), "kind": "oracle",
               "host_cores_available": len(os.sched_getaffinity(0)),
               "sample": f"all {n_req} requests of one step (all {g} positions, full V), "
                         f"{reps} times, of the same seeded bytes, {dt:.1f} s"}

    clocks = sampler.summary(w0, w1)
    others = None
    if rank == 0 and world == 1 and not args.no_other_configs:
        others = other_configs(spec, workloads, dev, peak)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": config_dict({"parallelism": f"replicas x{world}",
                                       "timing": "the step is one CUDA graph; value from K "
                                                 "replays without per-launch events; launch "
                                                 "durations from a replayed capture with "
                                                 "events around each library launch"}),
                "timing_spread": spread, "parity": parity,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(launches), "clocks": clocks,
                "tokens_per_s": float(n_acc.sum().item() + R) * args.steps * world / (ms / 1e3),
                "mean_accept_len": float(n_acc.float().mean().item()),
                "mean_emitted_per_request": float(n_acc.float().mean().item()) + 1.0,
                "other_configs": others}
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
