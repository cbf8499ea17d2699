"""Tensor-core projections (txl_qkv_proj, txl_r_proj) against the oracle's
fp64 projections of the same bf16 inputs.  Tolerance as for the bf16
attention: max|d| <= 1e-2 * max|ref| + 1e-3 (bf16 output rounding, fp32
accumulation over d)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl

pytestmark = pytest.mark.gpu


def tol(ref):
    return 1e-2 * float(np.abs(ref).max()) + 1e-3


def rand(*shape, std=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.empty(shape).normal_(0.0, std, generator=g).bfloat16()


@pytest.mark.parametrize("B,L,M,H", [
    (2, 128, 128, 8),     # the segment-128 workload's shape, 2 batch rows
    (1, 256, 0, 4),       # no memory yet
    (2, 128, 384, 16),    # d = 1024, memory longer than the segment
    (3, 384, 128, 4),     # several row tiles per source
])
def test_qkv_proj_matches_oracle(B, L, M, H):
    d = H * 64
    h, mem = rand(B, L, d, seed=1), rand(B, M, d, seed=2)
    w = rand(3 * d, d, std=0.05, seed=3)
    q, k, v = txl.qkv_proj(h.cuda(), mem.cuda(), w.cuda(), H)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    rq, rk, rv = oracle.qkv_proj(h, mem, w, H)
    for got, ref in ((q, rq), (k, rk), (v, rv)):
        g = got.float().cpu().double().numpy()
        assert g.shape == ref.shape
        assert np.abs(g - ref).max() <= tol(ref)


def test_qkv_proj_full_base512_shape():
    """The base-size workload's layer shapes (B=22, L=M=512, H=8)."""
    B, L, M, H = 22, 512, 512, 8
    d = H * 64
    h, mem = rand(B, L, d, seed=4), rand(B, M, d, seed=5)
    w = rand(3 * d, d, std=0.02, seed=6)
    q, k, v = txl.qkv_proj(h.cuda(), mem.cuda(), w.cuda(), H)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.qkv_proj(h, mem, w, H)
    for got, ref in ((q, rq), (k, rk), (v, rv)):
        assert np.abs(got.float().cpu().double().numpy() - ref).max() <= tol(ref)


@pytest.mark.parametrize("K,H", [(256, 8), (1024, 16), (3328, 16)])
def test_r_proj_matches_oracle(K, H):
    d = H * 64
    emb, w = rand(K, d, seed=7), rand(d, d, std=0.05, seed=8)
    r = txl.r_proj(emb.cuda(), w.cuda(), H)
    torch.cuda.synchronize()
    ref = oracle.r_proj(emb, w, H)
    assert np.abs(r.float().cpu().double().numpy() - ref).max() <= tol(ref)


def test_projections_reject_unsupported_sizes():
    H, d = 8, 512
    h = torch.zeros(1, 100, d, dtype=torch.bfloat16, device="cuda")  # L not a multiple of 128
    mem = torch.zeros(1, 128, d, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(3 * d, d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(txl.TxlError) as e:
        txl.qkv_proj(h, mem, w, H)
    assert e.value.code == -2


@pytest.mark.parametrize("B,L,M,H,h_heads,mem_start", [
    (22, 512, 512, 8, False, 0),    # the base-size workload's layer
    (1, 256, 0, 4, False, 0),       # no memory yet: r over L rows only
    (2, 128, 384, 16, True, 256),   # heads-layout input, ring memory read from row 256
])
def test_qkvr_proj_is_qkv_proj_and_r_proj_in_one_launch(B, L, M, H, h_heads, mem_start):
    """txl_qkvr_proj writes exactly (bit for bit) what txl_qkv_proj_ring and
    txl_r_proj write separately (same tiles, same accumulation order), and
    r_k matches the oracle's projection."""
    d = H * 64
    h, mem = rand(B, L, d, seed=11), rand(B, M, d, seed=12)
    w = rand(3 * d, d, std=0.03, seed=13)
    emb, wr = rand(M + L, d, seed=14), rand(d, d, std=0.03, seed=15)
    hd = h.cuda()
    if h_heads:
        hd = hd.view(B, L, H, 64).permute(0, 2, 1, 3).contiguous()
    q0, k0, v0 = txl.qkv_proj(hd, mem.cuda(), w.cuda(), H, mem_start=mem_start)
    r0 = txl.r_proj(emb.cuda(), wr.cuda(), H)
    q1, k1, v1, r1 = txl.qkvr_proj(hd, mem.cuda(), w.cuda(), emb.cuda(), wr.cuda(), H, mem_start=mem_start)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    for a, b in ((q0, q1), (k0, k1), (v0, v1), (r0, r1)):
        assert torch.equal(a, b)
    ref = oracle.r_proj(emb, wr, H)
    assert np.abs(r1.float().cpu().double().numpy() - ref).max() <= tol(ref)
