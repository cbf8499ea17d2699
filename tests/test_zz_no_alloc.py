"""txl_attn_fwd_noalloc against txl_attn_fwd_ws on two consecutive calls.

The no-alloc entry point runs the split-key path out of the library's static
device scratch; with a caller workspace the same kernels must give the same
bits.  This file is collected last so that it also runs after every other
GPU test has used the library on the same device."""
import pytest
import torch

import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # TXL_NOALLOC_SCRATCH_BYTES


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    shapes = [(1, 2, 128, 3000, 21), (2, 3, 200, 1500, 22)]  # both take the split-key path
    for B, H, L, M, seed in shapes:
        need = txl.attn_workspace_bytes(B, H, L, M, 64)
        assert 0 < need <= SCRATCH_BYTES
    outs = []
    for B, H, L, M, seed in shapes:  # two consecutive calls through the static scratch
        ci = W.random_call_inputs(B, H, L, M, 64, seed=seed)
        dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
        outs.append((dev, ci.scale, txl.attn_fwd_noalloc(*dev, scale=ci.scale)))
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    for (dev, scale, got), (B, H, L, M, _) in zip(outs, shapes):
        ws = torch.empty(txl.attn_workspace_bytes(B, H, L, M, 64), dtype=torch.uint8, device="cuda")
        ref = txl.attn_fwd_ws(*dev, ws, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_noalloc_without_split_matches_plain_entry():
    ci = W.random_call_inputs(2, 2, 256, 128, 64, seed=23)
    dev = [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]
    assert txl.attn_workspace_bytes(2, 2, 256, 128, 64) >= 0
    a = txl.attn_fwd_noalloc(*dev, scale=ci.scale)
    b = txl.attn_fwd(*dev, scale=ci.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_noalloc_rejects_calls_beyond_its_scratch():
    """Few items with a very long memory split into many units; once their
    partial results outgrow the static scratch the call is refused, not run.
    The split (and so the scratch a call needs) depends on this GPU's SM
    count, so the shape is searched for here, smallest first; finding none
    is a failure, not a skip."""
    found = None
    for M in (8000, 16000, 32000, 64000):
        for H in (8, 16, 24, 32, 40, 48, 64, 100, 140):
            if txl.attn_workspace_bytes(1, H, 128, M, 64) > SCRATCH_BYTES:
                found = (1, H, 128, M)
                break
        if found:
            break
    assert found, "no searched shape needs more than the static scratch"
    B, H, L, M = found
    q = torch.zeros(B, H, L, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(B, H, M + L, 64, device="cuda", dtype=torch.bfloat16)
    r = torch.zeros(M + L, H, 64, device="cuda", dtype=torch.bfloat16)
    u = torch.zeros(H, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(txl.TxlError) as e:
        txl.attn_fwd_noalloc(q, k, k, r, u, u, scale=0.125)
    assert e.value.code == -9
