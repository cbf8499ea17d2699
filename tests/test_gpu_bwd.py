"""Attention backward (txl_attn_bwd) against the oracle's gradients, which
are pinned to finite differences of the forward oracle: fp32 inputs within
1e-4*max|ref| + 1e-5, bf16 inputs within 1e-2*max|ref| + 1e-3 per gradient."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dr", "du", "dvb")


def check(ci, g, rtol, atol, **kw):
    d = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    got = txl.attn_bwd(*d, g.cuda(), ci.scale, **kw)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    ref = oracle.attn_bwd(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, g, **kw)
    for n in NAMES:
        r = ref[n]
        err = np.abs(got[n].cpu().double().numpy() - r).max()
        assert err <= rtol * np.abs(r).max() + atol, (n, err, np.abs(r).max())


@pytest.mark.parametrize("B,H,L,M,dh", [(1, 2, 8, 8, 16), (2, 3, 33, 20, 32), (1, 2, 70, 0, 64),
                                         (1, 1, 40, 90, 64),
                                         (1, 2, 20, 12, 128),    # d_h > 64: one query row per warp
                                         (1, 2, 35, 9, 18)])     # d_h not a multiple of 4
def test_f32_backward_matches_oracle(B, H, L, M, dh):
    ci = W.random_call_inputs(B, H, L, M, dh, dtype=torch.float32, std=0.5, seed=L + M)
    g = torch.randn(B, H, L, dh, generator=torch.Generator().manual_seed(1))
    check(ci, g, 1e-4, 1e-5)


def test_f32_backward_same_length():
    ci = W.random_call_inputs(1, 2, 24, 16, 32, dtype=torch.float32, std=0.5, seed=3)
    g = torch.randn(1, 2, 24, 32, generator=torch.Generator().manual_seed(2))
    check(ci, g, 1e-4, 1e-5, same_length=True, mem_len=16)


@pytest.mark.parametrize("L,M", [(128, 128), (100, 37)])
def test_bf16_backward_matches_oracle(L, M):
    ci = W.random_call_inputs(2, 2, L, M, 64, std=0.5, seed=7)
    g = torch.randn(2, 2, L, 64, generator=torch.Generator().manual_seed(3)).bfloat16()
    check(ci, g, 1e-2, 1e-3)


def test_backward_of_the_memory_rows_is_returned_not_propagated():
    """The memory's keys and values get gradients (a constant input still has
    them); q, u, v and R are unaffected by whether M rows exist beyond what
    the mask lets a query see."""
    ci = W.random_call_inputs(1, 1, 16, 16, 32, dtype=torch.float32, std=0.5, seed=5)
    g = torch.randn(1, 1, 16, 32, generator=torch.Generator().manual_seed(4))
    d = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    got = txl.attn_bwd(*d, g.cuda(), ci.scale)
    torch.cuda.synchronize()
    assert float(got["dk"][:, :, :16].abs().sum()) > 0 and float(got["dv"][:, :, :16].abs().sum()) > 0
