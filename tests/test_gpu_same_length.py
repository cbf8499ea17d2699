"""same_length attention (txl_attn_fwd_ex) against the oracle: fp32 within
1e-5, bf16 within 1e-2*max|ref| + 1e-3, the visibility picture read through
a one-hot probe, invisible keys provably unread, and the plain mask when the
context fits in mem_len."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu


def run(ci, mem_len, same_length=True):
    d = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    out = txl.attn_fwd(*d, ci.scale, same_length=same_length, mem_len=mem_len)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    return out


def ref(ci, mem_len):
    return oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, same_length=True,
                       mem_len=mem_len)


@pytest.mark.parametrize("B,H,L,M,mem_len", [
    (1, 2, 8, 8, 8), (2, 3, 33, 20, 20), (1, 2, 17, 5, 9), (1, 1, 40, 0, 7), (2, 2, 12, 30, 30)])
def test_f32_same_length_matches_oracle(B, H, L, M, mem_len):
    ci = W.random_call_inputs(B, H, L, M, 32, dtype=torch.float32, seed=L + M)
    got = run(ci, mem_len).cpu().double().numpy()
    assert np.abs(got - ref(ci, mem_len)).max() <= 1e-5


@pytest.mark.parametrize("B,H,L,M,mem_len", [
    (2, 2, 256, 256, 256),   # each query sees its 256 most recent keys
    (1, 3, 200, 300, 300),   # ragged query tail, memory not a tile multiple
    (1, 2, 128, 128, 384),   # memory still filling (M < mem_len)
    (1, 2, 384, 0, 128),     # no memory: a sliding window of 128
    (2, 1, 512, 512, 512),   # base-size shape, whole tiles skipped
])
def test_bf16_same_length_matches_oracle(B, H, L, M, mem_len):
    ci = W.random_call_inputs(B, H, L, M, 64, seed=B * 100 + L + M)
    got = run(ci, mem_len).float().cpu().double().numpy()
    r = ref(ci, mem_len)
    assert np.abs(got - r).max() <= 1e-2 * np.abs(r).max() + 1e-3


def test_same_length_picture_on_the_gpu():
    """fp32 one-hot probe: every score 0, so the output row is the
    probability row; M = mem_len = 3, L = 4 (each query sees 3 keys)."""
    M, L, dh = 3, 4, 8
    K = M + L
    q = torch.randn(1, 1, L, dh)
    k = torch.zeros(1, 1, K, dh)
    v = torch.zeros(1, 1, K, dh)
    for j in range(K):
        v[0, 0, j, j] = 1.0
    z = torch.zeros(K, 1, dh)
    ci = W.CallInputs(q, k, v, z, torch.zeros(1, dh), torch.randn(1, dh), 0.125)
    probs = run(ci, 3)[0, 0, :, :K].cpu().numpy()
    for i in range(L):
        vis = np.flatnonzero(probs[i] > 0)
        assert list(vis) == [i + 1, i + 2, i + 3]
        np.testing.assert_allclose(probs[i][vis], 1.0 / 3, atol=1e-6)


def test_bf16_invisible_keys_are_not_read():
    """Changing every key, value and position row a query may not see leaves
    its output bit-identical (masked entries and skipped tiles alike).  With
    M = mem_len = 256 and L = 384, query i sees keys i+1 .. 256+i and
    distances 0 .. 255; queries 256.. (the last two 128-row query tiles, which
    skip their first four key tiles) see no key below 257."""
    B, H, L, M, mem_len = 1, 2, 384, 256, 256
    ci = W.random_call_inputs(B, H, L, M, 64, seed=9)
    a = run(ci, mem_len).clone()
    k, v, r = ci.k.clone(), ci.v.clone(), ci.r_k.clone()
    k[:, :, :257] = 7.0
    v[:, :, :257] = -7.0
    r[:M + L - mem_len] = 5.0   # R rows of distances >= mem_len
    b = run(W.CallInputs(ci.q, k, v, r, ci.u, ci.vb, ci.scale), mem_len)
    assert torch.equal(a[:, :, 256:], b[:, :, 256:])
    # and the perturbation does reach the queries that see those keys
    assert not torch.equal(a[:, :, :256], b[:, :, :256])


def test_same_length_with_a_long_window_is_the_plain_mask():
    ci = W.random_call_inputs(2, 2, 256, 128, 64, seed=4)
    a = run(ci, 1000)
    b = run(ci, None, same_length=False)
    assert torch.equal(a, b)


def test_same_length_rejects_mem_len_below_M():
    ci = W.random_call_inputs(1, 1, 128, 128, 64, seed=1)
    with pytest.raises(txl.TxlError):
        run(ci, 64)
