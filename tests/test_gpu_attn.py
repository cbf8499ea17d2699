"""GPU parity of the attention kernels against the fp64 oracle, through the C ABI.

Tolerances: fp32 path max|d| <= 1e-5; bf16 inputs with fp32 accumulation
max|d| <= 1e-2 * max|ref| + 1e-3 (elementwise over the whole output, or over
the sampled (batch row, head) pairs at the full workload sizes).
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu


def bf16_tol(ref):
    return 1e-2 * float(np.nanmax(np.abs(ref))) + 1e-3


def run_gpu(ci, out=None):
    dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    o = txl.attn_fwd(*dev, scale=ci.scale, out=out)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    return o.float().cpu().double().numpy()


def check_bf16(ci, pairs=None):
    got = run_gpu(ci)
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, pairs=pairs)
    B, H = ci.q.shape[:2]
    sel = range(B * H) if pairs is None else pairs
    g = np.stack([got[p // H, p % H] for p in sel])
    r = np.stack([ref[p // H, p % H] for p in sel])
    assert np.isfinite(g).all()
    err = np.abs(g - r).max()
    assert err <= bf16_tol(r), f"max|d| = {err}, tol = {bf16_tol(r)}"
    return err


# ----------------------------------------------------------------- fp32 path
@pytest.mark.parametrize("M,L", [(8, 8), (3, 4), (0, 8), (0, 1), (37, 50), (5, 70)])
def test_f32_parity_tiny(M, L):
    wl = W.WORKLOADS["tiny_f32"].with_(M=M, L=L)
    ci, _, _ = W.first_call_inputs(wl)
    got = run_gpu(ci)
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)
    assert np.abs(got - ref).max() <= 1e-5


@pytest.mark.parametrize("dh", [16, 64, 100, 256])
def test_f32_parity_random(dh):
    ci = W.random_call_inputs(2, 3, 33, 20, dh, dtype=torch.float32, seed=dh)
    got = run_gpu(ci)
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)
    assert np.abs(got - ref).max() <= 1e-5


# ----------------------------------------------------------------- bf16 path
@pytest.mark.parametrize("B,H,L,M", [
    (1, 1, 128, 0),      # one tile, causal only
    (2, 2, 128, 128),    # memory tile + diagonal tile
    (1, 2, 200, 136),    # ragged query tail, memory not a tile multiple
    (2, 1, 77, 3),       # short, odd memory
    (1, 1, 1, 5),        # one query row
    (1, 2, 300, 0),      # several query tiles, no memory
    (2, 2, 256, 384),    # several tiles both ways
    (1, 1, 129, 1),      # query tail of one row
    (1, 3, 130, 1000),   # long memory, ragged
])
def test_bf16_parity_random_inputs(B, H, L, M):
    check_bf16(W.random_call_inputs(B, H, L, M, 64, seed=B * 1000 + L + M))


@pytest.mark.parametrize("B,H,L,M", [(2, 2, 128, 128), (1, 2, 200, 136), (3, 1, 64, 0)])
def test_bf16_parity_projected_inputs(B, H, L, M):
    wl = W.WORKLOADS["seg128_bf16"].with_(B=B, H=H, L=L, M=M)
    ci, _, _ = W.first_call_inputs(wl)
    check_bf16(ci)


def test_bf16_seg128_full_workload():
    """Segment-128 workload (B=16, H=8, L=M=128): every (b, h) pair."""
    ci, _, _ = W.first_call_inputs(W.WORKLOADS["seg128_bf16"])
    check_bf16(ci)


@pytest.mark.parametrize("name", ["base512_bf16", "large384_bf16", "longmem3200_bf16"])
def test_bf16_full_size_sampled(name):
    """Full-size first call of each large workload, in the launch configuration
    the benchmark times; the oracle checks a seeded sample of (b, h) pairs."""
    wl = W.WORKLOADS[name]
    ci, _, _ = W.first_call_inputs(wl)
    n = wl.B * wl.H
    rng = np.random.default_rng(7)
    pairs = sorted({0, n - 1, *rng.choice(n, size=4, replace=False).tolist()})
    check_bf16(ci, pairs=pairs)


@pytest.mark.parametrize("name,seg,layer", [("base512_bf16", 1, 5), ("base512_bf16", 2, 11),
                                            ("large384_bf16", 1, 17)])
def test_bf16_full_size_later_segment_and_layer(name, seg, layer):
    """A later call of the full-size chain, in the benchmark's launch
    configuration: segment ``seg`` (memories rolled by Tail_M through every
    earlier segment) and layer ``layer`` (its input the head-merged output of
    the layer below), on exactly the inputs that call saw.  The oracle checks
    a seeded sample of (b, h) pairs."""
    wl = W.WORKLOADS[name]
    dev = torch.device("cuda")
    dt = wl.torch_dtype
    params = W.make_params(wl)
    lws = [W.LayerWeights(*(getattr(lw, f).to(dev) for f in ("W_q", "W_k", "W_v", "W_r")))
           for lw in params.layers]
    mems = [m.to(device=dev, dtype=dt) for m in W.initial_memories(wl)]
    rks = [W.project_r(lw, wl.M, wl.L, wl.H, device=dev).to(dt) for lw in lws]
    u, vb = params.u.to(dev, dt), params.v.to(dev, dt)
    n_pairs = wl.B * wl.H
    pairs = sorted({0, n_pairs - 1,
                    *np.random.default_rng(seg * 100 + layer).choice(n_pairs, size=4, replace=False).tolist()})
    for s in range(seg + 1):
        h = W.segment_input(wl, s).to(device=dev, dtype=dt)
        for n in range(wl.layers):
            q, k, v = (x.to(dt) for x in W.project_qkv(lws[n], mems[n], h, wl.H))
            out = txl.attn_fwd(q, k, v, rks[n], u, vb, wl.scale)
            if (s, n) == (seg, layer):
                torch.cuda.synchronize()
                assert txl.sync_status() == 0
                got = out.float().cpu().double().numpy()
                ref = oracle.attn(q.cpu(), k.cpu(), v.cpu(), rks[n].cpu(), u.cpu(), vb.cpu(), wl.scale,
                                  pairs=pairs)
                g = np.stack([got[p // wl.H, p % wl.H] for p in pairs])
                r = np.stack([ref[p // wl.H, p % wl.H] for p in pairs])
                assert np.isfinite(g).all()
                assert np.abs(g - r).max() <= bf16_tol(r)
                return
            txl.mem_update(mems[n], h)
            h = W.merge_heads(out)
    raise AssertionError("the requested call was not reached")


def test_bf16_one_hot_probe_shows_mask_and_uniform_rows():
    """k = 0, u = 0, r_k = 0 and V_j = e_j: row i of the output is the
    probability row, 1/(M+i+1) on keys 0..M+i and exactly 0 past them."""
    M, L, dh = 20, 40, 64
    K = M + L
    z = torch.zeros
    v = torch.zeros(1, 1, K, dh)
    for j in range(K):
        v[0, 0, j, j] = 1.0
    ci = W.CallInputs(torch.randn(1, 1, L, dh).bfloat16(), z(1, 1, K, dh).bfloat16(),
                      v.bfloat16(), z(K, 1, dh).bfloat16(), z(1, dh).bfloat16(),
                      torch.randn(1, dh).bfloat16(), 0.125)
    got = run_gpu(ci)[0, 0]
    for i in range(L):
        row = got[i, :K]
        assert np.all(row[M + i + 1:] == 0.0)
        expect = float(torch.tensor(1.0 / (M + i + 1)).bfloat16())
        np.testing.assert_allclose(row[:M + i + 1], expect, rtol=1e-2)


def test_bf16_labelled_distance_probe():
    """q = k = u = 0, v_bias = e_0 and R row r holding its distance M+L-1-r in
    column 0: the score is scale * distance, so the log-probability ratio of
    two visible keys is scale * (distance difference).  One-hot V exposes the
    probabilities; this pins the relative shift on the GPU."""
    M, L, dh = 24, 36, 64
    K = M + L
    r = torch.zeros(K, 1, dh)
    r[:, 0, 0] = torch.arange(K - 1, -1, -1, dtype=torch.float32)
    vb = torch.zeros(1, dh); vb[0, 0] = 1.0
    v = torch.zeros(1, 1, K, dh)
    for j in range(K):
        v[0, 0, j, j] = 1.0
    z = torch.zeros
    scale = 0.05
    ci = W.CallInputs(z(1, 1, L, dh).bfloat16(), z(1, 1, K, dh).bfloat16(), v.bfloat16(),
                      r.bfloat16(), z(1, dh).bfloat16(), vb.bfloat16(), scale)
    got = run_gpu(ci)[0, 0]
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, scale)[0, 0]
    assert np.abs(got - ref).max() <= bf16_tol(ref)
    for i in range(L):
        p = got[i, :M + i + 1]
        # probabilities increase with distance (scale > 0): key 0 is farthest
        dist = M + i - np.arange(M + i + 1)
        assert np.corrcoef(np.log(p), dist)[0, 1] > 0.999


def test_bf16_deterministic():
    ci = W.random_call_inputs(2, 2, 256, 256, 64, seed=3)
    a = run_gpu(ci)
    b = run_gpu(ci)
    assert np.array_equal(a, b)


def test_bf16_timeout_injection_then_recovery():
    """A withheld internal signal makes the kernel's bounded waits expire: the
    call reports TXL_ERR_DEVICE_TIMEOUT through the status word, the GPU context
    stays usable and the next call is correct."""
    ci = W.random_call_inputs(1, 1, 64, 64, 64, seed=11)
    dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    txl.debug_inject(1)
    txl.attn_fwd(*dev, scale=ci.scale)
    assert txl.sync_status() == -6
    assert txl.sync_status() == 0  # cleared
    check_bf16(ci)


# ------------------------------------------------------- split-key workspace path
@pytest.mark.parametrize("B,H,L,M", [
    (1, 2, 128, 3000),    # two items, long memory: many splits
    (2, 3, 200, 1500),    # ragged query tail, two query tiles per (b, h)
    (1, 1, 64, 700),      # one item, short query tile
    (2, 2, 128, 1000),    # memory not a tile multiple
])
def test_bf16_split_keys_with_workspace(B, H, L, M):
    ci = W.random_call_inputs(B, H, L, M, 64, seed=B * 7 + M)
    need = txl.attn_workspace_bytes(B, H, L, M, 64)
    assert need > 0  # fewer items than SMs: the call splits the keys
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    got = txl.attn_fwd_ws(*dev, ws, scale=ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    got = got.float().cpu().double().numpy()
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= bf16_tol(ref)
    # the unsplit entry point agrees within the same tolerance
    plain = run_gpu(ci)
    assert np.abs(plain - ref).max() <= bf16_tol(ref)


def test_bf16_workspace_entry_full_size_long_memory():
    """The long-memory workload (B=8, H=16, L=128, M=3200: 128 items) through
    the workspace entry point, with whatever split the launch picks; the
    oracle checks a seeded sample of (b, h)."""
    wl = W.WORKLOADS["longmem3200_bf16"]
    ci, _, _ = W.first_call_inputs(wl)
    need = txl.attn_workspace_bytes(wl.B, wl.H, wl.L, wl.M, wl.dh)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    got = txl.attn_fwd_ws(*dev, ws, scale=ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    got = got.float().cpu().double().numpy()
    n = wl.B * wl.H
    pairs = sorted({0, n - 1, *np.random.default_rng(9).choice(n, size=4, replace=False).tolist()})
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, pairs=pairs)
    g = np.stack([got[p // wl.H, p % wl.H] for p in pairs])
    r = np.stack([ref[p // wl.H, p % wl.H] for p in pairs])
    assert np.abs(g - r).max() <= bf16_tol(r)


def test_bf16_workspace_errors():
    B, H, L, M = 1, 2, 128, 3000
    ci = W.random_call_inputs(B, H, L, M, 64, seed=5)
    dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    need = txl.attn_workspace_bytes(B, H, L, M, 64)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(txl.TxlError) as e:
        txl.attn_fwd_ws(*dev, small, scale=ci.scale)
    assert e.value.code == -7
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(txl.TxlError) as e:
        txl.attn_fwd_ws(*dev, big[16:], scale=ci.scale)  # not 256-byte aligned
    assert e.value.code == -7
    # a workspace overlapping the output
    nout = dev[0].numel() * 2
    buf = torch.empty(need + nout, dtype=torch.uint8, device="cuda")
    out = buf[need - 256: need - 256 + nout].view(torch.bfloat16).view(dev[0].shape)
    with pytest.raises(txl.TxlError) as e:
        txl.attn_fwd_ws(*dev, buf[:need], scale=ci.scale, out=out)
    assert e.value.code == -4
