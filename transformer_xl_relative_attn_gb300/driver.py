"""Multi-segment driver: rolls per-layer memories across consecutive segments
on one CUDA stream.

For each segment and each layer n, in order ("Transformer-XL" notes, zty624,
sections "Segment-Level Recurrence" and "Training and Inference": read the
segment, attend to memory + current tokens, append the new hidden states,
drop the oldest):

    q, k, v, r_k, u, v_bias = project(n, mems[n], h)     caller's projections
    out = txl_attn_fwd(q, k, v, r_k, u, v_bias, ...)      fused kernel
    txl_mem_update(mems[n], h)                            Tail_M, in place
    h = next_input(n, out)                                caller's layer body

Every memory is a dense [B, M, d] buffer that the driver updates in place,
so the memories stay resident in HBM across segments and no allocation
happens per segment.  The projections and whatever the caller runs between
layers are the caller's; the driver launches the attention and memory kernels
and nothing else.  ``run_segment`` can be captured into a CUDA graph when the
callbacks are capturable (static buffers, no host synchronisation).

With a second stream (``mem_stream``) each roll runs there instead: it starts
once its layer's inputs have been projected (just before that layer's
attention), and the same layer of the next segment waits for it before
projecting, so the HBM-bound rolls overlap the following attention calls while
every data dependency of the recurrence is kept.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch

from . import _lib


class SegmentDriver:
    def __init__(self, mems: Sequence[torch.Tensor], stream: torch.cuda.Stream | None = None,
                 mem_stream: torch.cuda.Stream | None = None):
        if not mems:
            raise ValueError("need one memory per layer")
        self.mems = list(mems)
        B, M, d = self.mems[0].shape
        for m in self.mems:
            if m.shape != (B, M, d) or not m.is_cuda or not m.is_contiguous():
                raise ValueError("memories must be contiguous CUDA tensors of one shape [B, M, d]")
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.mems[0].device)
        self.mem_stream = mem_stream
        self._rolled = [None] * len(self.mems)  # event after the last roll of each memory
        self.segments_done = 0

    @property
    def n_layers(self) -> int:
        return len(self.mems)

    def run_segment(self, h0: torch.Tensor,
                    project: Callable[[int, torch.Tensor, torch.Tensor], tuple],
                    next_input: Callable[[int, torch.Tensor], torch.Tensor],
                    outs: list | None = None) -> torch.Tensor:
        """Runs one segment through all layers; returns the last layer's
        next_input.  If ``outs`` is given, each layer's attention output is
        written into outs[n] (preallocated [B,H,L,dh]) instead of a new tensor."""
        h = h0
        with torch.cuda.stream(self.stream):
            for n, mem in enumerate(self.mems):
                if self._rolled[n] is not None:
                    self.stream.wait_event(self._rolled[n])
                q, k, v, r_k, u, vb, scale = project(n, mem, h)
                if self.mem_stream is not None:
                    projected = torch.cuda.Event()
                    projected.record(self.stream)
                out = _lib.attn_fwd(q, k, v, r_k, u, vb, scale,
                                    out=None if outs is None else outs[n], stream=self.stream)
                if self.mem_stream is None:
                    _lib.mem_update(mem, h, stream=self.stream)
                else:
                    self.mem_stream.wait_event(projected)
                    _lib.mem_update(mem, h, stream=self.mem_stream)
                    h.record_stream(self.mem_stream)  # h stays allocated until the roll read it
                    self._rolled[n] = torch.cuda.Event()
                    self._rolled[n].record(self.mem_stream)
                h = next_input(n, out)
        self.segments_done += 1
        return h

    def _wait_rolls(self) -> None:
        cur = torch.cuda.current_stream(self.mems[0].device)
        for ev in self._rolled:
            if ev is not None:
                cur.wait_event(ev)

    def state_dict(self) -> dict:
        """The only state is the per-layer memory (checkpoint/resume)."""
        self._wait_rolls()
        return {"mems": [m.detach().clone() for m in self.mems], "segments_done": self.segments_done}

    def load_state_dict(self, sd: dict) -> None:
        self._wait_rolls()
        for m, s in zip(self.mems, sd["mems"]):
            m.copy_(s)
        torch.cuda.synchronize(self.mems[0].device)  # later rolls see the restored memories
        self.segments_done = int(sd.get("segments_done", 0))
