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


def _push(mem: torch.Tensor, h: torch.Tensor, start: int, stream) -> int:
    """Ring-buffer update of one memory with the layer input h (either
    layout); returns the new ring start."""
    if mem.dim() == 4:
        B, H, M, dh = mem.shape
        return _lib.mem_ring_push(mem.view(B * H, M, dh), h.view(B * H, h.shape[2], dh), start, stream=stream)
    return _lib.mem_ring_push(mem, h, start, stream=stream)


def _roll(mem: torch.Tensor, h: torch.Tensor, stream, ext_len: int = 0) -> None:
    """Tail_M roll of one memory with the layer input h, in either layout:
    rows ([B, M, d] with [B, L, d]) or heads ([B, H, M, d_h] with
    [B, H, L, d_h], rolled as B*H independent rows of d_h elements)."""
    if mem.dim() == 4:
        B, H, M, dh = mem.shape
        _lib.mem_update(mem.view(B * H, M, dh), h.view(B * H, h.shape[2], dh), stream=stream,
                        ext_len=ext_len)
    else:
        _lib.mem_update(mem, h, stream=stream, ext_len=ext_len)


class AttnStack:
    """A stack of relative-attention layers over per-layer recurrence
    memories, every step in libtxl.so: for each segment and layer n

        q, k, v = txl_qkv_proj_ex(h, mems[n], W_qkv[n])     tensor-core projections
        txl_mem_update(mems[n], h)                           Tail_M, in place
        h = txl_attn_fwd(q, k, v, r_k[n], u[n], v[n])        fused attention

    ("Transformer-XL模型 核心源码阅读笔记", RelPartialLearnableMultiHeadAttn.forward
    and MemTransformerLM._update_mems; "Transformer-XL" notes, sections
    "Batched Tensor Contract" and "Segment-Level Recurrence").  Each layer's
    attention output is the next layer's input, kept in the heads layout
    [B, H, L, d_h] that the attention writes and the projections read; the
    output projection, residual, layer norm and feed-forward of a full layer
    are not part of this stack.  Layer 0's input arrives as rows [B, L, d];
    so layer 0's memory is rows [B, M, d] and every other memory is heads
    [B, H, M, d_h].  r_k[n] ([M+L, H, d_h]) depends on M and L only, so it is
    projected once, by the caller (txl_r_proj).

    Options of the source notes' MemTransformerLM: ``same_length`` (every
    query attends over the same number of keys, txl_attn_fwd_ex with mem_len
    = M), ``ext_len`` (the last ext_len rows of each segment stay out of the
    memory, txl_mem_update_ext), and ``reset_rows`` (per-row memory reset at
    document boundaries, txl_mem_reset).  With ``ring`` the memories are ring
    buffers sharing one start row: the projections read them through
    txl_qkv_proj_ring and txl_mem_ring_push writes each segment's L rows over
    the oldest ones instead of moving all M (``logical_mems`` gives the
    unrotated view; ring needs M and L multiples of 128 and ext_len = 0).

    The roll of mems[n] reads h after its projection has read mems[n].  On
    one stream that order is the launch order; with ``mem_stream`` each roll
    runs there, after an event recorded behind its projection, overlapping
    the layer's attention, and the stream waits for all rolls at the end of
    the segment (so the next segment, and whatever the caller launches after
    run_segment, sees the rolled memories and may reuse h0).  q, k and v are
    one set of buffers reused by every layer; each
    layer's output has its own buffer (the next layer's input and the source
    of its memory roll).
    """

    def __init__(self, w_qkv: Sequence[torch.Tensor], r_k: Sequence[torch.Tensor],
                 u: Sequence[torch.Tensor], v_bias: Sequence[torch.Tensor],
                 mems: Sequence[torch.Tensor], scale: float, n_head: int, seg_len: int,
                 stream: torch.cuda.Stream | None = None, same_length: bool = False,
                 ext_len: int = 0, ring: bool = False, mem_stream: torch.cuda.Stream | None = None):
        n = len(mems)
        if not (len(w_qkv) == len(r_k) == len(u) == len(v_bias) == n) or n == 0:
            raise ValueError("need one weight, r_k, u, v and memory per layer")
        m0 = mems[0]
        if m0.dim() != 3:
            raise ValueError("layer 0's memory must be rows [B, M, d]")
        B, M, d = m0.shape
        H = n_head
        if d % H:
            raise ValueError("d must be a multiple of n_head")
        dh = d // H
        for m in mems[1:]:
            if m.shape != (B, H, M, dh):
                raise ValueError("memories of layers >= 1 must be heads [B, H, M, d_h]")
        for m in mems:
            if not (m.is_cuda and m.is_contiguous() and m.dtype == torch.bfloat16):
                raise ValueError("memories must be contiguous bf16 CUDA tensors")
        self.w_qkv, self.r_k, self.u, self.v_bias = list(w_qkv), list(r_k), list(u), list(v_bias)
        self.mems = list(mems)
        self.scale, self.H, self.L = float(scale), H, int(seg_len)
        self.same_length, self.ext_len = bool(same_length), int(ext_len)
        self.ring, self.start = bool(ring), 0
        self.mem_stream = mem_stream
        if self.ring and (self.ext_len or int(seg_len) % 128 or m0.shape[1] % 128):
            raise ValueError("ring memories need ext_len = 0 and M, L multiples of 128")
        self.B, self.M, self.d, self.dh = B, M, d, dh
        dev = m0.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        L = self.L
        self.q = torch.empty((B, H, L, dh), **bf)
        self.k = torch.empty((B, H, M + L, dh), **bf)
        self.v = torch.empty((B, H, M + L, dh), **bf)
        self.outs = [torch.empty((B, H, L, dh), **bf) for _ in range(n)]
        self.segments_done = 0

    @property
    def n_layers(self) -> int:
        return len(self.mems)

    def run_segment(self, h0: torch.Tensor, trace: list | None = None,
                    out: torch.Tensor | None = None) -> torch.Tensor:
        """One segment through every layer; h0 is [B, L, d] bf16 on the device.
        Returns the last layer's attention output [B, H, L, d_h]: ``out`` if
        given, else a buffer of the stack that the next segment overwrites.
        With ``trace`` (tests), appends per layer the inputs each kernel saw
        and what it wrote."""
        if h0.shape != (self.B, self.L, self.d):
            raise ValueError(f"h0 must be [{self.B}, {self.L}, {self.d}]")
        h = h0
        with torch.cuda.stream(self.stream):
            for n, mem in enumerate(self.mems):
                rec = None
                if trace is not None:
                    rec = {"n": n, "h": h.clone(), "mem": mem.clone()}
                _lib.qkv_proj(h, mem, self.w_qkv[n], self.H, q=self.q, k=self.k, v=self.v,
                              stream=self.stream, mem_start=self.start if self.ring else 0)
                rs = self.stream
                if self.mem_stream is not None:
                    projected = torch.cuda.Event()
                    projected.record(self.stream)
                    self.mem_stream.wait_event(projected)
                    rs = self.mem_stream
                if self.ring:
                    new_start = _push(mem, h, self.start, rs)
                else:
                    _roll(mem, h, rs, self.ext_len)
                if self.mem_stream is not None and n == 0:
                    h.record_stream(self.mem_stream)  # the caller's h0 stays allocated for the roll
                dst = out if (out is not None and n == len(self.mems) - 1) else self.outs[n]
                o = _lib.attn_fwd(self.q, self.k, self.v, self.r_k[n], self.u[n], self.v_bias[n],
                                  self.scale, out=dst, stream=self.stream,
                                  same_length=self.same_length, mem_len=self.M)
                if rec is not None:
                    rec.update(q=self.q.clone(), k=self.k.clone(), v=self.v.clone(), out=o.clone())
                    trace.append(rec)
                h = o
            if self.mem_stream is not None:
                rolled = torch.cuda.Event()
                rolled.record(self.mem_stream)
                self.stream.wait_event(rolled)
        if self.ring:
            self.start = new_start
        self.segments_done += 1
        return h

    def logical_mems(self) -> list:
        """Copies of the memories in logical order (oldest row first)."""
        out = []
        for m in self.mems:
            ax = 1 if m.dim() == 3 else 2
            out.append(torch.roll(m, -self.start, dims=ax) if self.ring and self.start else m.clone())
        return out

    def reset_rows(self, flags: torch.Tensor) -> None:
        """Zeroes every layer's memory of the batch rows whose flag is set
        (their streams start a new document); other rows keep theirs."""
        with torch.cuda.stream(self.stream):
            for m in self.mems:
                _lib.mem_reset(m, flags, stream=self.stream)

    def state_dict(self) -> dict:
        """The per-layer memories (checkpoint/resume), with the ring start."""
        return {"mems": [m.detach().clone() for m in self.mems], "segments_done": self.segments_done,
                "start": self.start}

    def load_state_dict(self, sd: dict) -> None:
        for m, s in zip(self.mems, sd["mems"]):
            m.copy_(s)
        self.segments_done = int(sd.get("segments_done", 0))
        self.start = int(sd.get("start", 0))


class DecoderStack:
    """Full Transformer-XL decoder layers over per-layer recurrence memories
    ("Transformer-XL模型 核心源码阅读笔记": RelPartialLearnableDecoderLayer =
    RelPartialLearnableMultiHeadAttn then PositionwiseFF; MemTransformerLM keeps
    each layer's input as that layer's memory), every step in libtxl.so.  Per
    segment and layer n, with h the layer input [B, L, d] (rows):

      post-norm (pre_lnorm = False, the notes' default):
        q, k, v = txl_qkv_proj(h, mems[n])          roll mems[n] with h
        o   = txl_attn_fwd(q, k, v, r_k[n], u[n], v[n])          [B, H, L, d_h]
        h1  = LN1(h + o_net(o))                     txl_linear (heads input) + txl_layer_norm
        h   = LN2(h1 + W2 relu(W1 h1 + b1) + b2)    txl_linear x2 + txl_layer_norm
      pre-norm:
        q, k, v = txl_qkv_proj(LN1(h), LN1(mems[n]))
        h1  = h + o_net(o)                          residual fused into txl_linear
        h   = h1 + W2 relu(W1 LN2(h1) + b1) + b2

    ``layers[n]`` holds bf16 CUDA tensors: w_qkv [3d, d], w_o [d, d], ln1_g,
    ln1_b, ln2_g, ln2_b [d], w1 [d_inner, d], b1 [d_inner], w2 [d, d_inner],
    b2 [d] (nn.Linear layouts).  Memories are rows [B, M, d].  One stream
    orders every dependency; activations ping-pong between two buffers (a
    layer's input is dead once its memory has been rolled and its residuals
    read).
    """

    _keys = ("w_qkv", "w_o", "ln1_g", "ln1_b", "w1", "b1", "w2", "b2", "ln2_g", "ln2_b")

    def __init__(self, layers: Sequence[dict], r_k: Sequence[torch.Tensor], u: Sequence[torch.Tensor],
                 v_bias: Sequence[torch.Tensor], mems: Sequence[torch.Tensor], scale: float, n_head: int,
                 seg_len: int, pre_lnorm: bool = False, stream: torch.cuda.Stream | None = None,
                 same_length: bool = False, ext_len: int = 0, eps: float = 1e-5):
        n = len(mems)
        if not (len(layers) == len(r_k) == len(u) == len(v_bias) == n) or n == 0:
            raise ValueError("need one parameter set, r_k, u, v and memory per layer")
        B, M, d = mems[0].shape
        for m in mems:
            if m.shape != (B, M, d) or not m.is_cuda or not m.is_contiguous() or m.dtype != torch.bfloat16:
                raise ValueError("memories must be contiguous bf16 CUDA tensors [B, M, d]")
        for lp in layers:
            missing = [k for k in self._keys if k not in lp]
            if missing:
                raise ValueError(f"layer parameters missing {missing}")
        self.layers = [dict(lp) for lp in layers]
        self.r_k, self.u, self.v_bias, self.mems = list(r_k), list(u), list(v_bias), list(mems)
        self.scale, self.H, self.L, self.B, self.M, self.d = float(scale), n_head, int(seg_len), B, M, d
        self.dh = d // n_head
        self.d_inner = self.layers[0]["w1"].shape[0]
        self.pre_lnorm, self.same_length, self.ext_len, self.eps = bool(pre_lnorm), bool(same_length), int(ext_len), eps
        dev = mems[0].device
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        L, H, dh = self.L, self.H, self.dh
        self.q = torch.empty((B, H, L, dh), **bf)
        self.k = torch.empty((B, H, M + L, dh), **bf)
        self.v = torch.empty((B, H, M + L, dh), **bf)
        self.o = torch.empty((B, H, L, dh), **bf)
        self.h1 = torch.empty((B, L, d), **bf)
        self.f1 = torch.empty((B, L, self.d_inner), **bf)
        self.t = torch.empty((B, L, d), **bf)
        self.act = [torch.empty((B, L, d), **bf), torch.empty((B, L, d), **bf)]
        if self.pre_lnorm:
            self.hn = torch.empty((B, L, d), **bf)
            self.mn = torch.empty((B, M, d), **bf)
        self.segments_done = 0

    @property
    def n_layers(self) -> int:
        return len(self.mems)

    def run_segment(self, h0: torch.Tensor, trace: list | None = None,
                    out: torch.Tensor | None = None) -> torch.Tensor:
        """One segment through every layer; h0 [B, L, d] bf16 on the device.
        Returns the last layer's output [B, L, d] (``out`` if given, else a
        buffer the next segment overwrites).  ``trace`` (tests) collects the
        inputs and outputs of every step."""
        if h0.shape != (self.B, self.L, self.d):
            raise ValueError(f"h0 must be [{self.B}, {self.L}, {self.d}]")
        st, eps = self.stream, self.eps
        h = h0
        with torch.cuda.stream(st):
            for n, mem in enumerate(self.mems):
                lp = self.layers[n]
                rec = {"n": n, "h": h.clone(), "mem": mem.clone()} if trace is not None else None
                if self.pre_lnorm:
                    _lib.layer_norm(h, lp["ln1_g"], lp["ln1_b"], eps=eps, out=self.hn, stream=st)
                    _lib.layer_norm(mem, lp["ln1_g"], lp["ln1_b"], eps=eps, out=self.mn, stream=st)
                    _lib.qkv_proj(self.hn, self.mn, lp["w_qkv"], self.H, q=self.q, k=self.k, v=self.v, stream=st)
                else:
                    _lib.qkv_proj(h, mem, lp["w_qkv"], self.H, q=self.q, k=self.k, v=self.v, stream=st)
                _roll(mem, h, st, self.ext_len)
                _lib.attn_fwd(self.q, self.k, self.v, self.r_k[n], self.u[n], self.v_bias[n], self.scale,
                              out=self.o, stream=st, same_length=self.same_length, mem_len=self.M)
                last = n == len(self.mems) - 1
                dst = out if (out is not None and last) else self.act[(n + 1) % 2] if h is not self.act[(n + 1) % 2] \
                    else self.act[n % 2]
                if self.pre_lnorm:
                    _lib.linear(self.o, lp["w_o"], resid=h, out=self.h1, stream=st)
                    _lib.layer_norm(self.h1, lp["ln2_g"], lp["ln2_b"], eps=eps, out=self.t, stream=st)
                    _lib.linear(self.t, lp["w1"], bias=lp["b1"], relu=True, out=self.f1, stream=st)
                    _lib.linear(self.f1, lp["w2"], bias=lp["b2"], resid=self.h1, out=dst, stream=st)
                else:
                    _lib.linear(self.o, lp["w_o"], out=self.t, stream=st)
                    _lib.layer_norm(h, lp["ln1_g"], lp["ln1_b"], y=self.t, eps=eps, out=self.h1, stream=st)
                    _lib.linear(self.h1, lp["w1"], bias=lp["b1"], relu=True, out=self.f1, stream=st)
                    _lib.linear(self.f1, lp["w2"], bias=lp["b2"], out=self.t, stream=st)
                    _lib.layer_norm(self.h1, lp["ln2_g"], lp["ln2_b"], y=self.t, eps=eps, out=dst, stream=st)
                if rec is not None:
                    rec.update(q=self.q.clone(), k=self.k.clone(), v=self.v.clone(), o=self.o.clone(),
                               h1=self.h1.clone(), f1=self.f1.clone(), out=dst.clone())
                    if self.pre_lnorm:
                        rec.update(hn=self.hn.clone(), mn=self.mn.clone(), h1n=self.t.clone())
                    trace.append(rec)
                h = dst
        self.segments_done += 1
        return h

    def reset_rows(self, flags: torch.Tensor) -> None:
        """Zeroes every layer's memory of the flagged batch rows."""
        with torch.cuda.stream(self.stream):
            for m in self.mems:
                _lib.mem_reset(m, flags, stream=self.stream)

    def state_dict(self) -> dict:
        return {"mems": [m.detach().clone() for m in self.mems], "segments_done": self.segments_done}

    def load_state_dict(self, sd: dict) -> None:
        for m, s in zip(self.mems, sd["mems"]):
            m.copy_(s)
        self.segments_done = int(sd.get("segments_done", 0))
