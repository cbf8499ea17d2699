"""Decoder layers on the GPU (txl_linear, txl_layer_norm, DecoderStack)
against the oracle: each kernel on the inputs it saw, post- and pre-norm
stacks layer by layer, memories bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def tol(ref):
    return 1e-2 * float(np.abs(ref).max()) + 1e-3


def close(got, ref):
    g = got.float().cpu().double().numpy()
    assert g.shape == ref.shape
    assert np.abs(g - ref).max() <= tol(ref)


def rnd(*shape, std=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.empty(shape).normal_(0.0, std, generator=g).to(BF)


@pytest.mark.parametrize("B,T,K,N,heads,bias,relu,resid", [
    (2, 128, 256, 256, False, False, False, False),
    (2, 256, 512, 1024, False, True, True, False),    # first feed-forward layer
    (1, 384, 1024, 512, False, True, False, True),    # second layer with the residual
    (2, 128, 512, 512, True, False, False, False),    # o_net on a head-split attention output
    (8, 1024, 256, 2048, False, True, True, True),    # enough tiles for the 256-column tile width
    (8, 1024, 512, 512, True, False, False, True),    # 256 tiles of 128 x 128: the narrow width
])
def test_linear_matches_oracle(B, T, K, N, heads, bias, relu, resid):
    x = rnd(B, T, K, seed=1)
    w = rnd(N, K, std=K ** -0.5, seed=2)
    b = rnd(N, std=0.3, seed=3) if bias else None
    r = rnd(B, T, N, seed=4) if resid else None
    xin = W._split_heads(x.float(), K // 64).to(BF) if heads else x
    got = txl.linear(xin.cuda(), w.cuda(), bias=None if b is None else b.cuda(),
                     resid=None if r is None else r.cuda(), relu=relu)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    ref = oracle.linear(x, w, b)
    if relu:
        ref = np.maximum(ref, 0.0)
    if resid:
        ref = ref + r.double().numpy()
    close(got, ref)


@pytest.mark.parametrize("rows,d,with_y", [(300, 512, True), (64, 1024, False), (8, 256, True),
                                           (1000, 2048, True), (5, 768, False)])
def test_layer_norm_matches_oracle(rows, d, with_y):
    x = rnd(rows, d, std=2.0, seed=5)
    y = rnd(rows, d, seed=6) if with_y else None
    g = (1.0 + rnd(d, std=0.1, seed=7).float()).to(BF)
    b = rnd(d, std=0.1, seed=8)
    got = txl.layer_norm(x.cuda(), g.cuda(), b.cuda(), y=None if y is None else y.cuda())
    torch.cuda.synchronize()
    z = x.double() + (y.double() if y is not None else 0)
    close(got, oracle.layer_norm(z.numpy(), g, b))


def test_layer_norm_in_place():
    x = rnd(64, 512, seed=9).cuda()
    g, b = torch.ones(512, dtype=BF, device="cuda"), torch.zeros(512, dtype=BF, device="cuda")
    ref = txl.layer_norm(x, g, b)
    txl.layer_norm(x, g, b, out=x)
    torch.cuda.synchronize()
    assert torch.equal(ref, x)


WL = W.WORKLOADS["seg128_bf16"].with_(B=2, H=4, L=128, M=128, layers=2, segments=2)
D_INNER = 512


def make_stack(pre_lnorm):
    dev = torch.device("cuda")
    d, H, L, M = WL.d, WL.H, WL.L, WL.M
    layers = []
    for n in range(WL.layers):
        s = 100 * n
        layers.append({
            "w_qkv": rnd(3 * d, d, std=d ** -0.5, seed=s + 1), "w_o": rnd(d, d, std=d ** -0.5, seed=s + 2),
            "ln1_g": (1 + rnd(d, std=0.1, seed=s + 3).float()).to(BF), "ln1_b": rnd(d, std=0.1, seed=s + 4),
            "w1": rnd(D_INNER, d, std=d ** -0.5, seed=s + 5), "b1": rnd(D_INNER, std=0.1, seed=s + 6),
            "w2": rnd(d, D_INNER, std=D_INNER ** -0.5, seed=s + 7), "b2": rnd(d, std=0.1, seed=s + 8),
            "ln2_g": (1 + rnd(d, std=0.1, seed=s + 9).float()).to(BF), "ln2_b": rnd(d, std=0.1, seed=s + 10)})
    cpu_layers = layers
    layers = [{k: t.to(dev) for k, t in lp.items()} for lp in layers]
    emb = W.sinusoid(torch.arange(M + L - 1, -1, -1), d).to(dev, BF)
    r_k = [txl.r_proj(emb, rnd(d, d, std=d ** -0.5, seed=50 + n).to(dev), H) for n in range(WL.layers)]
    u = [rnd(H, WL.dh, std=0.1, seed=60).to(dev)] * WL.layers
    vb = [rnd(H, WL.dh, std=0.1, seed=61).to(dev)] * WL.layers
    mems = [rnd(WL.B, M, d, seed=70 + n).to(dev) for n in range(WL.layers)]
    st = txl.DecoderStack(layers, r_k, u, vb, mems, WL.scale, H, L, pre_lnorm=pre_lnorm)
    return st, cpu_layers, r_k, u, vb


@pytest.mark.parametrize("pre_lnorm", [False, True])
def test_decoder_stack_matches_oracle_step_by_step(pre_lnorm):
    st, lps, r_k, u, vb = make_stack(pre_lnorm)
    ref_mem = [m.cpu().view(torch.int16).numpy() for m in st.mems]
    trace = []
    for s in range(WL.segments):
        st.run_segment(W.segment_input(WL, s).cuda().to(BF), trace=trace)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    c = lambda t: t.cpu()
    for idx, rec in enumerate(trace):
        n, lp = rec["n"], lps[rec["n"]]
        assert np.array_equal(rec["mem"].cpu().view(torch.int16).numpy(), ref_mem[n])
        ref_mem[n] = oracle.mem_update(ref_mem[n], rec["h"].cpu().view(torch.int16).numpy(), WL.M)
        if idx > 0 and n > 0:
            assert torch.equal(trace[idx - 1]["out"], rec["h"])
        if pre_lnorm:
            close(rec["hn"], oracle.layer_norm(c(rec["h"]), lp["ln1_g"], lp["ln1_b"]))
            close(rec["mn"], oracle.layer_norm(c(rec["mem"]), lp["ln1_g"], lp["ln1_b"]))
            xin, min_ = c(rec["hn"]), c(rec["mn"])
        else:
            xin, min_ = c(rec["h"]), c(rec["mem"])
        rq, rk, rv = oracle.qkv_proj(xin, min_, lp["w_qkv"], WL.H)
        close(rec["q"], rq), close(rec["k"], rk), close(rec["v"], rv)
        ref_o = oracle.attn(c(rec["q"]), c(rec["k"]), c(rec["v"]), c(r_k[n]), c(u[n]), c(vb[n]), WL.scale)
        close(rec["o"], ref_o)
        vec = oracle.merge_heads(c(rec["o"]))
        close(rec["h1"], oracle.attn_block_out(c(rec["h"]), vec, lp["w_o"], lp["ln1_g"], lp["ln1_b"], pre_lnorm))
        close(rec["out"], oracle.pos_ff(c(rec["h1"]), lp["w1"], lp["b1"], lp["w2"], lp["b2"],
                                        lp["ln2_g"], lp["ln2_b"], pre_lnorm))
    for n, m in enumerate(st.mems):
        assert np.array_equal(m.cpu().view(torch.int16).numpy(), ref_mem[n])


def test_decoder_stack_checkpoint_resume_is_identical():
    st, *_ = make_stack(False)
    h = [W.segment_input(WL, s).cuda().to(BF) for s in range(3)]
    st.run_segment(h[0])
    sd = st.state_dict()
    a = st.run_segment(h[1]).clone()
    st.load_state_dict(sd)
    b = st.run_segment(h[1])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
