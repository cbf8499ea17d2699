"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module holds the input recipe only: the named shapes, the seeded random
draws, the sinusoid position table and the harness projections that turn
hidden states into per-head Q, K, V and R.  It holds none of the attention
arithmetic (no scores, mask, softmax or memory roll), so both the CUDA path
and the CPU oracle can consume what it produces without sharing any of the
method's code.

Recipe (all draws from one CPU ``torch.Generator`` seeded per workload):

* weights ``W_q, W_k, W_v, W_r`` are ``[d, d]`` per layer; hidden states and
  memories are ``N(0, act_std)``; the per-head biases ``u, v`` are ``[H, d_h]``
  and shared by all layers, as ``r_w_bias`` / ``r_r_bias`` are in
  "Transformer-XL模型 核心源码阅读笔记", section "Build the model"
  (MemTransformerLM._create_params);
* ``N(0, s)`` means standard deviation ``s`` (``torch.normal_(0, s)``), except
  that the tiny fp32 case draws its weights with variance ``1/d``;
* R is the sinusoid table of the distances ``M+L-1 .. 0`` (sin half first,
  then cos half, not interleaved: PositionalEmbedding in the same notes)
  times ``W_r``;
* projections run in fp32 (TF32 off) and are cast once to the workload dtype;
  the GPU and the oracle consume those identical cast tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    dh: int
    L: int
    M: int
    dtype: str          # "f32" or "bf16"
    layers: int
    segments: int
    seed: int
    w_std: float        # weight standard deviation
    uv_std: float       # u, v standard deviation
    act_std: float = 1.0

    @property
    def d(self) -> int:
        return self.H * self.dh

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dh)

    def visible_pairs(self) -> int:
        """Visible (query, key) pairs per (batch row, head): L*M + L(L+1)/2."""
        return self.L * self.M + self.L * (self.L + 1) // 2

    def attn_flops(self) -> int:
        """Algorithmic FLOPs of one attention call: content, position and PV
        contractions (2*d_h each) over the visible pairs only."""
        return 6 * self.dh * self.B * self.H * self.visible_pairs()

    def mem_update_bytes(self) -> int:
        """Compulsory bytes of one Tail_M roll: M rows read, M rows written."""
        es = 4 if self.dtype == "f32" else 2
        return 2 * self.B * self.M * self.d * es

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # fp32 single layer; the M=3/L=4 mask case and the M=0 case are derived
    # from it in the tests.
    "tiny_f32": Workload("tiny_f32", B=1, H=2, dh=16, L=8, M=8, dtype="f32",
                         layers=1, segments=1, seed=0,
                         w_std=1.0 / math.sqrt(32), uv_std=0.1),
    "seg128_bf16": Workload("seg128_bf16", B=16, H=8, dh=64, L=128, M=128,
                            dtype="bf16", layers=1, segments=4, seed=1,
                            w_std=0.02, uv_std=0.02),
    "base512_bf16": Workload("base512_bf16", B=22, H=8, dh=64, L=512, M=512,
                             dtype="bf16", layers=12, segments=3, seed=2,
                             w_std=0.02, uv_std=0.02),
    "large384_bf16": Workload("large384_bf16", B=16, H=16, dh=64, L=384, M=384,
                              dtype="bf16", layers=18, segments=2, seed=3,
                              w_std=0.02, uv_std=0.02),
    "longmem3200_bf16": Workload("longmem3200_bf16", B=8, H=16, dh=64, L=128,
                                 M=3200, dtype="bf16", layers=1, segments=8,
                                 seed=4, w_std=0.02, uv_std=0.02),
}


def sinusoid(pos: torch.Tensor, demb: int) -> torch.Tensor:
    """Sinusoid table [len(pos), demb]: sin(pos*f) for the first half of the
    columns, cos(pos*f) for the second, f_k = 10000^(-2k/demb)."""
    inv_freq = 1.0 / (10000.0 ** (torch.arange(0.0, demb, 2.0, dtype=torch.float64) / demb))
    ang = pos.to(torch.float64)[:, None] * inv_freq[None, :]
    return torch.cat([ang.sin(), ang.cos()], dim=-1).to(torch.float32)


@dataclass
class LayerWeights:
    W_q: torch.Tensor
    W_k: torch.Tensor
    W_v: torch.Tensor
    W_r: torch.Tensor


@dataclass
class Params:
    layers: list
    u: torch.Tensor   # [H, dh] fp32
    v: torch.Tensor   # [H, dh] fp32


def generator(wl: Workload, stream: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed * 1000003 + stream)
    return g


def _normal(shape, std, g):
    return torch.empty(shape, dtype=torch.float32).normal_(0.0, std, generator=g)


def make_params(wl: Workload, layers: int | None = None) -> Params:
    g = generator(wl, 1)
    nl = wl.layers if layers is None else layers
    d = wl.d
    lw = [LayerWeights(*(_normal((d, d), wl.w_std, g) for _ in range(4))) for _ in range(nl)]
    u = _normal((wl.H, wl.dh), wl.uv_std, g)
    v = _normal((wl.H, wl.dh), wl.uv_std, g)
    return Params(lw, u, v)


def initial_memories(wl: Workload, layers: int | None = None, M: int | None = None) -> list:
    """Per-layer memories [B, M, d] ~ N(0, act_std), fp32."""
    g = generator(wl, 2)
    nl = wl.layers if layers is None else layers
    m = wl.M if M is None else M
    return [_normal((wl.B, m, wl.d), wl.act_std, g) for _ in range(nl)]


def segment_input(wl: Workload, seg: int, L: int | None = None) -> torch.Tensor:
    """Layer-0 hidden state of segment ``seg``: [B, L, d] ~ N(0, act_std), fp32."""
    g = generator(wl, 100 + seg)
    return _normal((wl.B, wl.L if L is None else L, wl.d), wl.act_std, g)


def _split_heads(x: torch.Tensor, H: int) -> torch.Tensor:
    B, T, d = x.shape
    return x.reshape(B, T, H, d // H).permute(0, 2, 1, 3).contiguous()


def merge_heads(o: torch.Tensor) -> torch.Tensor:
    """[B, H, L, dh] -> [B, L, H*dh] (heads concatenated per position)."""
    B, H, L, dh = o.shape
    return o.permute(0, 2, 1, 3).reshape(B, L, H * dh).contiguous()


def _mm32(x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        return torch.matmul(x.to(torch.float32), w.to(device=x.device, dtype=torch.float32))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def project_qkv(lw: LayerWeights, mem: torch.Tensor, h: torch.Tensor, H: int):
    """Harness projections of one layer: Q from the current segment only, K and V
    from memory rows then current rows ("Transformer-XL" notes, zty624,
    section "Batched Tensor Contract").  Memory and current rows are projected
    separately and written into the two row ranges of K and V, so no hidden
    state concatenation is formed.  Returns fp32 q [B,H,L,dh], k, v [B,H,M+L,dh]."""
    B, L, d = h.shape
    M = mem.shape[1]
    q = _split_heads(_mm32(h, lw.W_q), H)
    k = torch.empty((B, H, M + L, d // H), dtype=torch.float32, device=h.device)
    v = torch.empty_like(k)
    if M > 0:
        k[:, :, :M] = _split_heads(_mm32(mem, lw.W_k), H)
        v[:, :, :M] = _split_heads(_mm32(mem, lw.W_v), H)
    k[:, :, M:] = _split_heads(_mm32(h, lw.W_k), H)
    v[:, :, M:] = _split_heads(_mm32(h, lw.W_v), H)
    return q, k, v


def position_sequence(M: int, L: int, clamp_len: int | None = None) -> torch.Tensor:
    """The positions of the relative table, klen-1 down to 0 (klen = M+L),
    optionally clamped from above at ``clamp_len`` as MemTransformerLM._forward
    does before the positional embedding ("Transformer-XL模型 核心源码阅读笔记",
    section "Build the model": pos_seq.clamp_(max=clamp_len) when clamp_len > 0;
    here any clamp_len >= 0 is applied, 0 included).  fp64."""
    pos = torch.arange(M + L - 1, -1, -1, dtype=torch.float64)
    if clamp_len is not None:
        pos = pos.clamp(max=float(clamp_len))
    return pos


def project_r(lw: LayerWeights, M: int, L: int, H: int, device="cpu",
              clamp_len: int | None = None) -> torch.Tensor:
    """R_k [M+L, H, dh], row r <-> distance M+L-1-r (fp32); with clamp_len,
    every distance beyond it uses the embedding of clamp_len."""
    d = lw.W_r.shape[0]
    pos = position_sequence(M, L, clamp_len)
    emb = sinusoid(pos, d).to(device)
    return _mm32(emb, lw.W_r).reshape(M + L, H, d // H).contiguous()


@dataclass
class CallInputs:
    """Everything one attention call consumes, already in the workload dtype."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    r_k: torch.Tensor
    u: torch.Tensor
    vb: torch.Tensor
    scale: float

    @property
    def shape(self):
        B, H, L, dh = self.q.shape
        return B, H, L, self.k.shape[2] - L, dh


def call_inputs(wl: Workload, lw: LayerWeights, params: Params, mem: torch.Tensor,
                h: torch.Tensor, r_k32: torch.Tensor | None = None) -> CallInputs:
    """Project one layer's inputs and cast them once to the workload dtype."""
    dt = wl.torch_dtype
    q, k, v = project_qkv(lw, mem, h, wl.H)
    M, L = mem.shape[1], h.shape[1]
    if r_k32 is None:
        r_k32 = project_r(lw, M, L, wl.H, device=h.device)
    dev = h.device
    return CallInputs(q.to(dt), k.to(dt), v.to(dt), r_k32.to(dt),
                      params.u.to(device=dev, dtype=dt), params.v.to(device=dev, dtype=dt),
                      wl.scale)


def first_call_inputs(wl: Workload, B: int | None = None) -> tuple:
    """Inputs of layer 0, segment 0 of a workload (optionally fewer batch rows),
    plus the layer-0 memory and hidden state they came from (workload dtype)."""
    w = wl if B is None else wl.with_(B=B)
    params = make_params(w, layers=1)
    mem = initial_memories(w, layers=1)[0]
    h = segment_input(w, 0)
    ci = call_inputs(w, params.layers[0], params, mem, h)
    return ci, mem.to(w.torch_dtype), h.to(w.torch_dtype)


def random_call_inputs(B: int, H: int, L: int, M: int, dh: int, dtype=torch.bfloat16,
                       std: float = 1.0, bias_std: float = 0.5, seed: int = 0) -> CallInputs:
    """Direct N(0, std) draws for every attention input (no projections), cast
    once to ``dtype``.  With std = 1 and scale = 1/sqrt(d_h) the scores spread
    over several units, so the softmax is far from uniform and a wrong score
    shows in the output."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    K = M + L

    def n(*shape, s=std):
        return torch.empty(shape, dtype=torch.float32).normal_(0.0, s, generator=g).to(dtype)

    return CallInputs(n(B, H, L, dh), n(B, H, K, dh), n(B, H, K, dh), n(K, H, dh),
                      n(H, dh, s=bias_std), n(H, dh, s=bias_std), 1.0 / math.sqrt(dh))
