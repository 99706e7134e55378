"""Device-resident draft -> verify loop.

One iteration is the whole token-level hot path of "[DeepSeek-6] DSpark": the Markov head's
serial proposal (section 3 and section 4 "Markov Head"), the target normalisers, the TV
confidence labels and their prefix survival (section 5, section 6), the hardware-aware prefix
scheduler's lengths (section 6), and lossless rejection verification of the scheduled prefixes
(speculative sampling with the residual / bonus draw). The token each request emits at the end
of iteration t (its residual or bonus draw) is the anchor x_0 of iteration t + 1; iteration t
reads slice t of the pre-drawn uniforms. The logit tensors stay fixed across iterations (the
models that would produce new logits are outside this library).

Every step is a call into libspecmarkov (argument marshalling only), and the iterations can be
captured into one CUDA graph so that no host round trip separates them.
"""
from __future__ import annotations

import torch

from . import spec as S


class SpecLoop:
    """`iterations` chained draft -> verify iterations over fixed logits.

    U [R, gamma, V] and target [R, gamma + 1, V] (bf16 or fp32), W1 / W2 [V, rank], anchors0
    [R] int32, uniforms u_draft / u_accept [iters, R, gamma] and u_resid [iters, R] fp32,
    sps [Bmax + 1] fp64 (index = batch size B). With schedule=False every request verifies
    all gamma positions (no confidence pass, no scheduler). `allowed` (optional, [R, ceil(V/32)]
    32-bit words) restricts every draft position to the allowed tokens (grammar-masked
    drafting), in the proposal, the confidence pass and the residual alike.

    async_schedule=True is the production form of the scheduler ("[DeepSeek-6] DSpark",
    section 7): iteration t still ranks its own candidates by its own survival, but the batch
    size it fills is the Theta-optimal one of iteration t - 2 (dynamic top-K). The first two
    iterations have no such history and use their own Theta optimum. One scheduler launch per
    iteration both selects and records the Theta optimum for iteration t + 2 (batch_opt).

    flat=True (with a scheduler) verifies the flattened batch of section 7: the scheduled rows
    are packed into B = sum_r (1 + l_r) consecutive rows with per-request offsets, the target
    normalisers are packed alike, and rejection verification reads the packed rows. The
    packing copy stands in for a target model that writes only the B scheduled rows; the
    outputs equal the padded loop's bit for bit."""

    def __init__(self, U, target, W1, W2, anchors0, u_draft, u_accept, u_resid, temperature,
                 sps=None, *, iterations=None, schedule=True, allowed=None,
                 async_schedule=False, flat=False):
        R, gamma, V = U.shape
        self.R, self.gamma, self.V = R, gamma, V
        self.iters = int(iterations if iterations is not None else u_draft.shape[0])
        self.U, self.target, self.W1, self.W2 = U, target, W1, W2
        self.u_draft, self.u_accept, self.u_resid = u_draft, u_accept, u_resid
        self.temperature = float(temperature)
        self.sps = sps
        self.allowed = allowed
        self.schedule = bool(schedule) and sps is not None
        self.async_schedule = self.schedule and bool(async_schedule)
        self.flat = self.schedule and bool(flat)
        self.rank = 0 if W1 is None else int(W1.shape[1])
        dev = U.device
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        n = self.iters
        self.anchors = torch.empty(n + 1, R, **i32)
        self.anchors[0].copy_(anchors0)
        self.draft_tokens = torch.empty(n, R, gamma, **i32)
        self.draft_logp = torch.empty(R, gamma, **f32)
        self.draft_stats = torch.empty(R, gamma, 2, **f32)
        self.target_stats = torch.empty(R * (gamma + 1), 2, **f32)
        self.conf = torch.empty(n, R, gamma, **f32)
        self.survival = torch.empty(n, R, gamma, **f32)
        self.lengths = torch.empty(n, R, **i32)
        self.batch = torch.empty(n, **i32)
        # Theta-optimal batch of iteration t >= 2 in async mode (for t < 2 it is batch[t])
        self.batch_opt = torch.empty(n, **i32)
        self.theta = torch.empty(n, dtype=torch.float64, device=dev)
        self.accept_len = torch.empty(n, R, **i32)
        self.out_tokens = torch.empty(n, R, gamma + 1, **i32)
        if self.flat:
            self.offsets = torch.empty(R + 1, **i32)
            self.packed_target = torch.empty(R * (gamma + 1), V, dtype=target.dtype, device=dev)
            self.packed_stats = torch.empty(R * (gamma + 1), 2, **f32)
        # one workspace large enough for every step, reserved before any capture
        self.ws = S.Workspace(device=dev)
        self.ws.reserve(int(S.lib().spec_workspace_bytes(S.SPEC_OP_ALL, R, gamma, V, self.rank)))
        self.graph = None

    def iteration(self, t: int, stream=None):
        """Enqueue iteration t on `stream` (the current stream by default)."""
        ws, T = self.ws, self.temperature
        a_t = self.anchors[t]
        S.spec_markov_propose(self.U, self.W1, self.W2, a_t, self.u_draft[t], T,
                              draft_tokens=self.draft_tokens[t], draft_logp=self.draft_logp,
                              draft_stats=self.draft_stats, workspace=ws, stream=stream,
                              allowed=self.allowed)
        S.spec_target_stats(self.target, T, stats=self.target_stats, workspace=ws, stream=stream)
        lengths = None
        if self.schedule:
            S.spec_tv_confidence(self.U, self.target, self.W1, self.W2, a_t,
                                 self.draft_tokens[t], T, draft_stats=self.draft_stats,
                                 target_stats=self.target_stats, conf=self.conf[t],
                                 survival=self.survival[t], workspace=ws, stream=stream,
                                 allowed=self.allowed)
            out = dict(lengths=self.lengths[t], B_out=self.batch[t:t + 1],
                       theta_out=self.theta[t:t + 1], workspace=ws, stream=stream)
            if self.async_schedule and t >= 2:
                # iterations 0 and 1 chose their own optimum, so it sits in `batch`
                hist = self.batch if t < 4 else self.batch_opt
                S.spec_schedule_prefix(self.survival[t], self.sps, capacity=hist[t - 2:t - 1],
                                       B_opt_out=self.batch_opt[t:t + 1], **out)
            else:
                S.spec_schedule_prefix(self.survival[t], self.sps, **out)
            lengths = self.lengths[t]
        if self.flat:
            # the flattened verify batch: B packed target rows and their normalisers
            S.spec_flat_layout(lengths, self.gamma, offsets=self.offsets, markers=False,
                               workspace=ws, stream=stream)
            tv = self.target.view(self.R, self.gamma + 1, self.V)
            S.spec_flat_pack(tv, lengths, self.offsets, out=self.packed_target, workspace=ws,
                             stream=stream)
            S.spec_flat_pack(self.target_stats.view(self.R, self.gamma + 1, 2), lengths,
                             self.offsets, out=self.packed_stats, workspace=ws, stream=stream)
            S.spec_verify_rejection_flat(self.packed_target, self.U, self.W1, self.W2, a_t,
                                         self.draft_tokens[t], self.draft_logp, self.draft_stats,
                                         self.u_accept[t], self.u_resid[t], T, lengths,
                                         self.offsets, target_stats=self.packed_stats,
                                         accept_len=self.accept_len[t],
                                         out_tokens=self.out_tokens[t],
                                         next_anchor=self.anchors[t + 1], workspace=ws,
                                         stream=stream, allowed=self.allowed)
            return
        S.spec_verify_rejection(self.target, self.U, self.W1, self.W2, a_t, self.draft_tokens[t],
                                self.draft_logp, self.draft_stats, self.u_accept[t],
                                self.u_resid[t], T, lengths, target_stats=self.target_stats,
                                accept_len=self.accept_len[t], out_tokens=self.out_tokens[t],
                                next_anchor=self.anchors[t + 1], workspace=ws, stream=stream,
                                allowed=self.allowed)

    def run(self, first: int = 0, last: int | None = None, stream=None):
        """Iterations first..last-1, enqueued eagerly. The loop state is anchors[first] and the
        iteration index (which selects the uniform slice), so a loop stopped after iteration t
        resumes exactly with run(t + 1, ...), given the same anchors and uniforms."""
        last = self.iters if last is None else last
        for t in range(first, last):
            self.iteration(t, stream)

    def capture(self, first: int = 0, last: int | None = None):
        """Record iterations first..last-1 into one CUDA graph (replay with replay())."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(first, last)
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    def emitted_tokens(self) -> torch.Tensor:
        """Tokens emitted per iteration and request: the accepted prefix plus one draw."""
        return self.accept_len + 1
