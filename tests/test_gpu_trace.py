"""Per-launch tracing through the C ABI (spec_trace_events): caller-owned CUDA events record
around each library launch of a kernel class, both for eager launches and for launches captured
into a CUDA graph (then every replay records them again)."""
import ctypes

import pytest
import torch

from draft_sampling_verification_markov_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spec():
    import __graft_entry__
    __graft_entry__.build()
    from draft_sampling_verification_markov_gb300 import spec as s
    return s


def _attach(spec, kclass, n, stream):
    b = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for x in b + e:
        x.record(stream)
    torch.cuda.synchronize()
    bh = (ctypes.c_void_p * n)(*[x.cuda_event for x in b])
    eh = (ctypes.c_void_p * n)(*[x.cuda_event for x in e])
    assert spec.lib().spec_trace_events(kclass, bh, eh, n) == 0
    return b, e, (bh, eh)


@pytest.mark.parametrize("captured", [False, True])
def test_trace_events_time_the_proposal_launch(spec, captured):
    wl = W.markov_rejection("cuda", R=130, gamma=3, V=4096, rank=128, seed=9)
    ws = spec.Workspace(device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())  # the inputs are drawn on the current stream
    run = lambda: spec.spec_markov_propose(wl.U, wl.W1, wl.W2, wl.anchors, wl.u_draft, 1.0,
                                           workspace=ws, stream=stream)
    run()                                           # sizes the workspace before any capture
    torch.cuda.synchronize()
    kc = spec.SPEC_KCLASS_PROPOSE
    b, e, keep = _attach(spec, kc, 8, stream)
    try:
        if captured:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run()
            count = spec.lib().spec_trace_count(kc)
            with torch.cuda.stream(stream):
                g.replay()
        else:
            run()
            count = spec.lib().spec_trace_count(kc)
        torch.cuda.synchronize()
    finally:
        spec.lib().spec_trace_events(kc, None, None, 0)
    # bf16 weights on the tensor cores: the whole proposal (three positions, two request
    # groups) is one persistent launch
    assert count == 1
    times = [b[i].elapsed_time(e[i]) for i in range(count)]
    assert all(t > 0 for t in times)
    assert ws.status() == 0
