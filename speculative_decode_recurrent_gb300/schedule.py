"""Decode-step schedules over several GDN layers, built from the library calls.

A decode step runs, for every layer in order, the verify of its draft block; the
accept of the step's accepted counts and the periodic flush follow.  A layer's accept
and flush are needed only by that layer's next verify, one step later ("The inference
stack behind OCRia", section "Making speculative verification cheaper": the checkpoint
is rewritten only at the periodic flush, and the rollback is a length update), so
they may run beside the verifies of the later layers.  Three orders of the same work:

* ``enqueue_overlap`` -- the verify of every layer on the current stream; the accept
  and flush of layer l on one of ``n_side`` side streams, forked after layer l's
  verify; the step ends with a join of the side streams;
* ``enqueue_three_call`` -- verify, accept, flush of each layer in order on the
  current stream;
* ``enqueue_fused`` -- verify_fold + accept_fold of each layer on the current stream
  (the flush folded into the next verify).

All three may be captured in a CUDA graph (the side streams fork from and join the
capturing stream).  They only enqueue library calls; every step runs in the kernels.
The optional hooks ``before(l)`` / ``after(l)`` run on the host right before layer
l's verify is enqueued and right after it, on the current stream (e.g. to wait for
that layer's inputs to arrive, or to start copying its outputs out).
"""
from __future__ import annotations

import torch


class StepSchedule:
    """Enqueues one decode step over ``layers`` (ReplayLayer objects)."""

    def __init__(self, layers, n_side: int = 2, device=None):
        self.layers = list(layers)
        self.sides = [torch.cuda.Stream(device=device) for _ in range(n_side)]
        self.fork = [torch.cuda.Event() for _ in self.layers]

    def enqueue_overlap(self, blocks, accepted, outs, marks=None, before=None, after=None):
        """blocks[l]: dict of device draft tensors (q, k, v, g, beta); accepted[l]:
        device int32 [B]; outs[l]: device fp32 [B, T, H, dv].  ``marks`` (two timing
        events) bracket the run of verifies on the current stream."""
        main = torch.cuda.current_stream()
        if marks is not None:
            marks[0].record()
        for l, layer in enumerate(self.layers):
            b = blocks[l]
            if before is not None:
                before(l)
            layer.verify(b["q"], b["k"], b["v"], b["g"], b["beta"], outs[l])
            if after is not None:
                after(l)
            side = self.sides[l % len(self.sides)]
            self.fork[l].record(main)
            side.wait_event(self.fork[l])
            with torch.cuda.stream(side):
                layer.accept(accepted[l])
                layer.flush(force=False)
        if marks is not None:
            marks[1].record()
        for side in self.sides:
            main.wait_stream(side)

    def enqueue_three_call(self, blocks, accepted, outs, events=None, before=None, after=None):
        """``events[l]`` (four timing events, optional) bracket layer l's calls."""
        for l, layer in enumerate(self.layers):
            b = blocks[l]
            if before is not None:
                before(l)
            if events is not None:
                events[l][0].record()
            layer.verify(b["q"], b["k"], b["v"], b["g"], b["beta"], outs[l])
            if after is not None:
                after(l)
            if events is not None:
                events[l][1].record()
            layer.accept(accepted[l])
            if events is not None:
                events[l][2].record()
            layer.flush(force=False)
            if events is not None:
                events[l][3].record()

    def enqueue_fused(self, blocks, accepted, outs, events=None, before=None, after=None):
        for l, layer in enumerate(self.layers):
            b = blocks[l]
            if before is not None:
                before(l)
            if events is not None:
                events[l][0].record()
            layer.verify_fold(b["q"], b["k"], b["v"], b["g"], b["beta"], outs[l])
            if after is not None:
                after(l)
            if events is not None:
                events[l][1].record()
            layer.accept_fold(accepted[l])
            if events is not None:
                events[l][2].record()
                events[l][3].record()

    def enqueue(self, mode, blocks, accepted, outs, **kw):
        return {"overlap": self.enqueue_overlap, "three_call": self.enqueue_three_call,
                "fused": self.enqueue_fused}[mode](blocks, accepted, outs, **kw)
