"""Ring-buffer memory (txl_mem_ring_push, txl_qkv_proj_ring, AttnStack with
ring=True): the logical memory equals the oracle's Tail_M roll bit for bit,
projections through the ring equal projections of the unrotated memory bit
for bit, and a ring stack reproduces the copying stack exactly."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("B,M,d,Ls", [
    (2, 384, 64, [128, 128, 128, 128, 256]),   # wraps, then a push of L < M across the end
    (1, 100, 24, [30, 30, 30, 50, 7]),        # odd sizes: scalar and 8-byte paths
    (3, 256, 512, [128, 512, 128]),           # L >= M refills the ring from row 0
])
def test_ring_push_matches_tail_m(B, M, d, Ls):
    g = torch.Generator().manual_seed(M + d)
    mem0 = torch.randn(B, M, d, generator=g).to(BF)
    ring = mem0.cuda()
    ref = bits(mem0)
    start = 0
    for L in Ls:
        h = torch.randn(B, L, d, generator=g).to(BF)
        start = txl.mem_ring_push(ring, h.cuda(), start)
        ref = oracle.mem_update(ref, bits(h), M)
        torch.cuda.synchronize()
        assert txl.sync_status() == 0
        logical = torch.roll(ring, -start, dims=1)
        assert np.array_equal(bits(logical), ref)


@pytest.mark.parametrize("start", [0, 128, 256])
def test_projection_through_the_ring_is_exact(start):
    g = torch.Generator().manual_seed(start + 1)
    B, H, L, M = 2, 8, 128, 384
    d = H * 64
    h = torch.randn(B, L, d, generator=g).to(BF).cuda()
    logical = torch.randn(B, M, d, generator=g).to(BF).cuda()
    ring = torch.roll(logical, start, dims=1).contiguous()   # logical row t at (start + t) % M
    w = (torch.randn(3 * d, d, generator=g) * 0.03).to(BF).cuda()
    a = txl.qkv_proj(h, logical, w, H)
    b = txl.qkv_proj(h, ring, w, H, mem_start=start)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_ring_rejects_unaligned_start():
    B, H, L, M = 1, 4, 128, 256
    d = H * 64
    z = torch.zeros(B, L, d, dtype=BF, device="cuda")
    m = torch.zeros(B, M, d, dtype=BF, device="cuda")
    w = torch.zeros(3 * d, d, dtype=BF, device="cuda")
    with pytest.raises(txl.TxlError):
        txl.qkv_proj(z, m, w, H, mem_start=64)


def make(ring, mem_stream=None):
    wl = W.WORKLOADS["seg128_bf16"].with_(B=2, H=4, L=128, M=384, layers=2, segments=5)
    dev = torch.device("cuda")
    p = W.make_params(wl)
    H, d, L, M = wl.H, wl.d, wl.L, wl.M
    w_qkv = [torch.cat([lw.W_q.t(), lw.W_k.t(), lw.W_v.t()]).contiguous().to(dev, BF) for lw in p.layers]
    emb = W.sinusoid(torch.arange(M + L - 1, -1, -1), d).to(dev, BF)
    r_k = [txl.r_proj(emb, lw.W_r.t().contiguous().to(dev, BF), H) for lw in p.layers]
    u, vb = [p.u.to(dev, BF)] * wl.layers, [p.v.to(dev, BF)] * wl.layers
    m0 = W.initial_memories(wl)
    mems = [m0[0].to(dev, BF)] + [W._split_heads(m, H).to(dev, BF) for m in m0[1:]]
    return wl, txl.AttnStack(w_qkv, r_k, u, vb, mems, wl.scale, H, L, ring=ring, mem_stream=mem_stream)


def test_ring_stack_reproduces_the_copying_stack():
    wl, a = make(False)
    _, b = make(True)
    for s in range(wl.segments):
        h0 = W.segment_input(wl, s).cuda().to(BF)
        oa = a.run_segment(h0).clone()
        ob = b.run_segment(h0).clone()
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), s
        for x, y in zip(a.logical_mems(), b.logical_mems()):
            assert torch.equal(x, y)
    assert b.start == (wl.segments * wl.L) % wl.M


@pytest.mark.parametrize("ring", [False, True])
def test_rolls_on_a_second_stream_change_nothing(ring):
    """The rolls (or ring pushes) on their own stream, overlapping the
    attention, give bit-identical outputs and memories."""
    wl, a = make(ring)
    _, b = make(ring, mem_stream=torch.cuda.Stream())
    for s in range(wl.segments):
        h0 = W.segment_input(wl, s).cuda().to(BF)
        oa = a.run_segment(h0).clone()
        ob = b.run_segment(h0).clone()
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), s
    for x, y in zip(a.logical_mems(), b.logical_mems()):
        assert torch.equal(x, y)
