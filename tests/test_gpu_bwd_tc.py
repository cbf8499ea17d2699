"""Tensor-core backward (txl_attn_bwd_ws: bf16, d_h = 64) against the
oracle's gradients, which are pinned to finite differences of the forward
oracle (tests/test_oracle_pins.py).  Tolerance per gradient: 1e-2*max|ref| +
1e-3, the bf16 bound of the forward (P and dS are rounded to bf16 before
their products, as the forward rounds P)."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dr", "du", "dvb")


def _dev(ci):
    return [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]


def _close(name, got, ref):
    err = np.abs(got - ref).max()
    tol = 1e-2 * np.abs(ref).max() + 1e-3
    assert err <= tol, (name, float(err), float(tol), float(np.abs(ref).max()))


def check(ci, g, names=NAMES):
    got = txl.attn_bwd(*_dev(ci), g.cuda(), ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    ref = oracle.attn_bwd(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, g)
    for n in names:
        _close(n, got[n].cpu().double().numpy(), ref[n])


@pytest.mark.parametrize("B,H,L,M", [
    (1, 2, 128, 128),   # one query tile, memory of two key tiles
    (2, 2, 100, 37),    # ragged query tile, memory not a multiple of 64
    (1, 1, 200, 0),     # no memory: causal attention with a relative bias
    (1, 2, 64, 300),    # long memory, one short query tile
    (2, 3, 257, 64),    # three query tiles, the last one row long
    (1, 1, 384, 200),   # several items per CTA-sized sweep, odd tile counts
])
def test_bf16_tc_backward_matches_oracle(B, H, L, M):
    ci = W.random_call_inputs(B, H, L, M, 64, std=0.5, seed=11 + L + M)
    g = torch.randn(B, H, L, 64, generator=torch.Generator().manual_seed(5)).bfloat16()
    check(ci, g)


def test_tc_and_cuda_core_paths_agree():
    """Both entry points compute the same gradients: the tensor-core passes
    round P and dS to bf16, the CUDA-core kernel keeps them in fp32."""
    ci = W.random_call_inputs(2, 2, 160, 96, 64, std=0.5, seed=3)
    g = torch.randn(2, 2, 160, 64, generator=torch.Generator().manual_seed(6)).bfloat16().cuda()
    a = txl.attn_bwd(*_dev(ci), g, ci.scale, tensor_cores=True)
    b = txl.attn_bwd(*_dev(ci), g, ci.scale, tensor_cores=False)
    torch.cuda.synchronize()
    for n in NAMES:
        x, y = a[n].double(), b[n].double()
        assert float((x - y).abs().max()) <= 1e-2 * float(y.abs().max()) + 1e-3, n


def test_workspace_is_required_and_checked():
    ci = W.random_call_inputs(1, 1, 64, 64, 64, std=0.5, seed=4)
    g = torch.randn(1, 1, 64, 64).bfloat16().cuda()
    need = txl.attn_bwd_workspace_bytes(1, 1, 64, 64, 64)
    assert need > 0
    assert txl.attn_bwd_workspace_bytes(1, 1, 64, 64, 64, same_length=True) == 0
    assert txl.attn_bwd_workspace_bytes(1, 1, 64, 64, 32) == 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(txl.TxlError) as e:
        txl.attn_bwd(*_dev(ci), g, ci.scale, workspace=small)
    assert e.value.code == -7


def test_repeated_calls_give_the_same_dq_dk_dv():
    """dq, dk and dv are written once per element (no atomics): bit-identical
    across calls; dr, du, dvb are zeroed by every call before accumulating."""
    ci = W.random_call_inputs(1, 2, 130, 70, 64, std=0.5, seed=8)
    g = torch.randn(1, 2, 130, 64, generator=torch.Generator().manual_seed(2)).bfloat16().cuda()
    a = txl.attn_bwd(*_dev(ci), g, ci.scale)
    b = txl.attn_bwd(*_dev(ci), g, ci.scale)
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
    for n in ("dr", "du", "dvb"):
        assert float((a[n] - b[n]).abs().max()) <= 1e-5 * float(a[n].abs().max()) + 1e-6, n


@pytest.mark.parametrize("name,pairs", [("base512_bf16", [(0, 0), (13, 5), (21, 7)])])
def test_full_size_sampled_pairs(name, pairs):
    """The bench workload's first call at full size: dq, dk, dv of sampled
    (b, h) pairs against the oracle run on those pairs alone."""
    wl = W.WORKLOADS[name]
    ci, _, _ = W.first_call_inputs(wl)
    B, H, L = ci.q.shape[:3]
    g = torch.randn(B, H, L, 64, generator=torch.Generator().manual_seed(7)).bfloat16()
    got = txl.attn_bwd(*_dev(ci), g.cuda(), ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    for b, h in pairs:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attn_bwd(ci.q[sl], ci.k[sl], ci.v[sl], ci.r_k[:, h:h + 1], ci.u[h:h + 1], ci.vb[h:h + 1],
                              ci.scale, g[sl])
        for n in ("dq", "dk", "dv"):
            _close(f"{n}[{b},{h}]", got[n][b:b + 1, h:h + 1].cpu().double().numpy(), ref[n])


def test_batch_summed_gradients_of_a_reduced_batch():
    """dR, du and dv_bias are sums over the batch and all pairs: a two-row
    batch of the bench workload's shape (L = M = 512, H = 8), in full."""
    wl = W.WORKLOADS["base512_bf16"]
    ci, _, _ = W.first_call_inputs(wl, B=2)
    g = torch.randn(2, wl.H, wl.L, 64, generator=torch.Generator().manual_seed(9)).bfloat16()
    check(ci, g, names=("dr", "du", "dvb", "dq"))


def _lse_bound(ci):
    """Per-row bound on |lse_gpu - lse_ref| in log2 units: the scores carry
    the bf16 rounding of (q+u)c, (q+v)c (relative 2^-9 per element) and the
    f16 rounding of the position term (2^-11); a log-sum-exp moves by at most
    the largest score error, bounded here with a factor 2 of margin."""
    q, k, r, u, vb = (t.double() for t in (ci.q, ci.k, ci.r_k, ci.u, ci.vb))
    qu = (q + u[None, :, None, :]).norm(dim=-1)                  # [B,H,L]
    qv = (q + vb[None, :, None, :]).norm(dim=-1)
    kn = k.norm(dim=-1).amax(dim=-1)                              # [B,H]
    rn = r.norm(dim=-1).amax(dim=0)                               # [H]
    s_max = qu * kn[:, :, None] + qv * rn[None, :, None]
    return (2.0 ** -8) * ci.scale * 1.4426950408889634 * s_max + 1e-4


@pytest.mark.parametrize("B,H,L,M", [(1, 2, 128, 128), (2, 2, 100, 37), (1, 1, 200, 0)])
def test_forward_lse_matches_oracle(B, H, L, M):
    ci = W.random_call_inputs(B, H, L, M, 64, std=0.5, seed=21 + L + M)
    d = _dev(ci)
    out0 = txl.attn_fwd(*d, scale=ci.scale)
    out, lse = txl.attn_fwd_lse(*d, scale=ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    assert torch.equal(out, out0)  # the same kernel, plus one store per row
    _, sc = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, want_scores=True)
    m = sc.max(axis=-1, keepdims=True)
    ref = (m[..., 0] + np.log(np.exp(sc - m).sum(axis=-1))) * 1.4426950408889634
    err = np.abs(lse.cpu().double().numpy() - ref)
    assert (err <= _lse_bound(ci).numpy()).all(), float(err.max())


@pytest.mark.parametrize("B,H,L,M", [(1, 2, 128, 128), (2, 2, 100, 37), (1, 1, 200, 0), (2, 3, 257, 64)])
def test_backward_from_saved_forward_state_matches_oracle(B, H, L, M):
    """txl_attn_bwd_saved: the gradients from the forward's saved out and lse
    (no recomputed forward) against the oracle."""
    ci = W.random_call_inputs(B, H, L, M, 64, std=0.5, seed=31 + L + M)
    d = _dev(ci)
    out, lse = txl.attn_fwd_lse(*d, scale=ci.scale)
    g = torch.randn(B, H, L, 64, generator=torch.Generator().manual_seed(5)).bfloat16()
    got = txl.attn_bwd(*d, g.cuda(), ci.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    ref = oracle.attn_bwd(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, g)
    for n in NAMES:
        _close(n, got[n].cpu().double().numpy(), ref[n])


def test_saved_state_entries_reject_bad_arguments():
    ci = W.random_call_inputs(1, 1, 64, 64, 64, std=0.5, seed=4)
    d = _dev(ci)
    out, lse = txl.attn_fwd_lse(*d, scale=ci.scale)
    g = torch.randn(1, 1, 64, 64).bfloat16().cuda()
    with pytest.raises(ValueError):
        txl.attn_bwd(*d, g, ci.scale, out=out)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(txl.TxlError) as e:
        txl.attn_bwd(*d, g, ci.scale, out=out, lse=lse, workspace=small)
    assert e.value.code == -7
    f32 = W.random_call_inputs(1, 1, 16, 16, 64, dtype=torch.float32, std=0.5, seed=4)
    with pytest.raises(txl.TxlError) as e:
        txl.attn_fwd_lse(*_dev(f32), scale=f32.scale)
    assert e.value.code == -2


def test_gradients_complete_for_work_queued_after_the_call():
    """The passes overlap on the GPU (the key-major pass starts on the SMs the
    query-major pass leaves) but the call's last launch completes after both:
    stream work queued right after the call, with no host synchronisation,
    sees every gradient final."""
    ci = W.random_call_inputs(2, 3, 257, 64, 64, std=0.5, seed=12)
    d = _dev(ci)
    g = torch.randn(2, 3, 257, 64, generator=torch.Generator().manual_seed(3)).bfloat16().cuda()
    ref = txl.attn_bwd(*d, g, ci.scale)
    torch.cuda.synchronize()
    grads = {n: torch.full_like(ref[n], float("nan")) for n in NAMES}
    got = txl.attn_bwd(*d, g, ci.scale, grads=grads)
    copies = {n: got[n].clone() for n in NAMES}  # queued on the same stream, no sync in between
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    for n in ("dq", "dk", "dv"):
        assert torch.equal(copies[n], ref[n]), n
    for n in ("dr", "du", "dvb"):
        assert float((copies[n] - ref[n]).abs().max()) <= 1e-5 * float(ref[n].abs().max()) + 1e-6, n
