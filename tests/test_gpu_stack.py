"""AttnStack (projections, Tail_M rolls and attention all in libtxl.so, layer
outputs fed to the next layer in the heads layout) against the oracle: every
projection and attention call matches the oracle on the inputs that call
saw, every memory a call saw is the oracle's Tail_M roll of the earlier
segments (bit-exact, in either layout), and a checkpoint taken between
segments resumes to identical results."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu

WL = W.WORKLOADS["seg128_bf16"].with_(B=2, H=4, L=128, M=128, layers=3, segments=3)
BF = torch.bfloat16


def tol(ref):
    return 1e-2 * float(np.abs(ref).max()) + 1e-3


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy()


def rows(x):
    """[B, T, d] as is; [B, H, T, d_h] -> [B, T, H*d_h]."""
    if x.dim() == 3:
        return x
    B, H, T, dh = x.shape
    return x.permute(0, 2, 1, 3).reshape(B, T, H * dh)


def make_stack(same_length=False, ext_len=0):
    dev = torch.device("cuda")
    p = W.make_params(WL)
    H, d, L, M = WL.H, WL.d, WL.L, WL.M
    # the library's nn.Linear layout: output = input W^T
    w_qkv = [torch.cat([lw.W_q.t(), lw.W_k.t(), lw.W_v.t()]).contiguous().to(dev, BF) for lw in p.layers]
    emb = W.sinusoid(torch.arange(M + L - 1, -1, -1), d).to(dev, BF)
    r_k = [txl.r_proj(emb, lw.W_r.t().contiguous().to(dev, BF), H) for lw in p.layers]
    u = [p.u.to(dev, BF)] * WL.layers
    vb = [p.v.to(dev, BF)] * WL.layers
    m0 = W.initial_memories(WL)
    mems = [m0[0].to(dev, BF)] + [W._split_heads(m, H).to(dev, BF) for m in m0[1:]]
    return (txl.AttnStack(w_qkv, r_k, u, vb, mems, WL.scale, H, L, same_length=same_length,
                          ext_len=ext_len), w_qkv, r_k, u, vb)


@pytest.mark.parametrize("same_length,ext_len,reset", [(False, 0, False), (True, 32, True)])
def test_stack_calls_and_memories_match_oracle(same_length, ext_len, reset):
    """The second case adds the MemTransformerLM options: same_length
    attention, ext_len rolls, and a per-row reset of batch row 1 before the
    third segment."""
    stack, w_qkv, r_k, u, vb = make_stack(same_length, ext_len)
    M = WL.M
    ref_mem = [bits(m) for m in stack.mems]
    trace = []
    flags = torch.tensor([False, True])
    for s in range(WL.segments):
        if reset and s == 2:
            stack.reset_rows(flags.cuda())
        h0 = W.segment_input(WL, s).cuda().to(BF)
        stack.run_segment(h0, trace=trace)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    assert len(trace) == WL.segments * WL.layers
    for idx, c in enumerate(trace):
        n = c["n"]
        if reset and idx == 2 * WL.layers:  # the reset before segment 2
            ref_mem = [oracle.mem_reset(m, flags.numpy()) for m in ref_mem]
        # the memory this call saw is the oracle's roll of the earlier segments
        assert np.array_equal(bits(c["mem"]), ref_mem[n])
        mem, h = c["mem"], c["h"]
        if mem.dim() == 4:
            B, H, _, dh = mem.shape
            nxt = oracle.mem_update(bits(mem).reshape(B * H, M, dh), bits(h).reshape(B * H, -1, dh), M,
                                    ext_len=ext_len)
            ref_mem[n] = nxt.reshape(B, H, M, dh)
        else:
            ref_mem[n] = oracle.mem_update(bits(mem), bits(h), M, ext_len=ext_len)
        # projections on the inputs the call saw
        rq, rk, rv = oracle.qkv_proj(rows(h).cpu(), rows(mem).cpu(), w_qkv[n].cpu(), WL.H)
        for got, ref in ((c["q"], rq), (c["k"], rk), (c["v"], rv)):
            g = got.float().cpu().double().numpy()
            assert np.abs(g - ref).max() <= tol(ref), n
        # attention on the q, k, v the call saw
        cpu = [t.cpu() for t in (c["q"], c["k"], c["v"], r_k[n], u[n], vb[n])]
        ref = oracle.attn(*cpu, WL.scale, same_length=same_length, mem_len=M)
        got = c["out"].float().cpu().double().numpy()
        assert np.abs(got - ref).max() <= tol(ref), n
    # each layer's input is the previous layer's output
    for a, b in zip(trace, trace[1:]):
        if b["n"] > 0:
            assert torch.equal(a["out"], b["h"])
    for n, m in enumerate(stack.mems):
        assert np.array_equal(bits(m), ref_mem[n])


def test_stack_checkpoint_resume_is_identical():
    stack, *_ = make_stack()
    h = [W.segment_input(WL, s).cuda().to(BF) for s in range(3)]
    stack.run_segment(h[0])
    sd = stack.state_dict()
    a = stack.run_segment(h[1]).clone()
    mem_a = [m.clone() for m in stack.mems]
    stack.load_state_dict(sd)
    assert stack.segments_done == 1
    b = stack.run_segment(h[1])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    for x, y in zip(mem_a, stack.mems):
        assert torch.equal(x, y)


def test_heads_layout_projection_matches_rows_layout():
    """txl_qkv_proj_ex reading h and mem in the heads layout gives exactly the
    result of the rows layout on the same values."""
    g = torch.Generator().manual_seed(5)
    B, H, L, M = 2, 8, 256, 128
    d = H * 64
    h = torch.empty(B, L, d).normal_(0, 1, generator=g).to(BF)
    mem = torch.empty(B, M, d).normal_(0, 1, generator=g).to(BF)
    w = torch.empty(3 * d, d).normal_(0, 0.03, generator=g).to(BF)
    hs = [x.cuda() for x in (h, mem, w)]
    q0, k0, v0 = txl.qkv_proj(hs[0], hs[1], hs[2], H)
    q1, k1, v1 = txl.qkv_proj(W._split_heads(h, H).cuda(), W._split_heads(mem, H).cuda(), hs[2], H)
    q2, k2, v2 = txl.qkv_proj(hs[0], W._split_heads(mem, H).cuda(), hs[2], H)
    torch.cuda.synchronize()
    for a, b, c in ((q0, q1, q2), (k0, k1, k2), (v0, v1, v2)):
        assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("clamp_len", [100, 0])
def test_stack_with_clamp_len_matches_oracle(clamp_len):
    """clamp_len ("Transformer-XL模型 核心源码阅读笔记", section "Build the model",
    MemTransformerLM._forward: pos_seq.clamp_(max=clamp_len) before the
    positional embedding): every distance beyond clamp_len takes the position
    embedding of clamp_len.  It changes only the position table the layer's
    r_k is projected from, so the stack runs unchanged on a clamped r_k: its
    rows for distances >= clamp_len come out bit-identical, and every call
    matches the oracle on the inputs it saw."""
    stack, w_qkv, r_k_plain, u, vb = make_stack()
    p = W.make_params(WL)
    H, d, L, M = WL.H, WL.d, WL.L, WL.M
    emb = W.sinusoid(W.position_sequence(M, L, clamp_len), d).cuda().to(BF)
    r_k = [txl.r_proj(emb, lw.W_r.t().contiguous().cuda().to(BF), H) for lw in p.layers]
    stack.r_k = r_k
    torch.cuda.synchronize()
    far = M + L - 1 - clamp_len          # rows 0..far hold distances >= clamp_len
    for r in r_k:
        assert all(torch.equal(r[i], r[far]) for i in range(far + 1))
        if far + 1 < M + L:
            assert not torch.equal(r[far], r[far + 1])
    trace = []
    for s in range(2):
        stack.run_segment(W.segment_input(WL, s).cuda().to(BF), trace=trace)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    differs = False
    for c in trace:
        n = c["n"]
        cpu = [t.cpu() for t in (c["q"], c["k"], c["v"], r_k[n], u[n], vb[n])]
        ref = oracle.attn(*cpu, WL.scale)
        got = c["out"].float().cpu().double().numpy()
        assert np.abs(got - ref).max() <= tol(ref), n
        plain = oracle.attn(*cpu[:3], r_k_plain[n].cpu(), *cpu[4:], WL.scale)
        differs |= np.abs(plain - ref).max() > tol(ref)
    assert differs  # the clamp is visible in the result
