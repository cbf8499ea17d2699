"""GPU Tail_M memory roll against the oracle: bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl

pytestmark = pytest.mark.gpu


def bits(t):
    t = t.contiguous().cpu()
    return t.view(torch.int16).numpy() if t.element_size() == 2 else t.view(torch.int32).numpy()


@pytest.mark.parametrize("B,M,L,d,dtype", [
    (2, 8, 8, 32, torch.float32),        # M = L
    (3, 12, 5, 64, torch.bfloat16),      # L < M, M not a multiple of L
    (2, 5, 12, 64, torch.bfloat16),      # L > M
    (8, 3200, 128, 1024, torch.bfloat16),  # long-memory workload shape
    (22, 512, 512, 512, torch.bfloat16),   # base-size workload shape
    (1, 7, 3, 5, torch.bfloat16),        # odd row bytes: scalar path
    (2, 9, 2, 6, torch.float32),         # 24-byte rows: 8-byte path
    (1, 100, 1, 8, torch.bfloat16),      # L = 1: one long chain per column
])
def test_tail_m_bit_exact(B, M, L, d, dtype):
    g = torch.Generator().manual_seed(B * 131 + M + L)
    mem = torch.randn(B, M, d, generator=g).to(dtype)
    hid = torch.randn(B, L, d, generator=g).to(dtype)
    expect = oracle.mem_update(bits(mem), bits(hid), M)
    dm = mem.cuda()
    txl.mem_update(dm, hid.cuda())
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    assert np.array_equal(bits(dm), expect)


def test_tail_m_m0_noop():
    mem = torch.zeros(2, 0, 8, device="cuda", dtype=torch.bfloat16)
    txl.mem_update(mem, torch.ones(2, 4, 8, device="cuda", dtype=torch.bfloat16))
    assert mem.numel() == 0


def test_tail_m_repeated_rolls_match_oracle():
    """Four consecutive segments rolled in place equal four oracle rolls."""
    B, M, L, d = 4, 40, 16, 64
    g = torch.Generator().manual_seed(5)
    mem = torch.randn(B, M, d, generator=g).bfloat16()
    ref = bits(mem)
    dm = mem.cuda()
    for s in range(4):
        h = torch.randn(B, L, d, generator=g).bfloat16()
        ref = oracle.mem_update(ref, bits(h), M)
        txl.mem_update(dm, h.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(dm), ref)


def test_tail_m_rejects_overlap():
    flat = torch.zeros(400, device="cuda", dtype=torch.bfloat16)
    mems = flat[0:160].view(1, 20, 8)
    hids = flat[80:112].view(1, 4, 8)   # inside the memory buffer
    with pytest.raises(txl.TxlError) as e:
        txl.mem_update(mems, hids)
    assert e.value.code == -4


@pytest.mark.parametrize("B,M,L,d,ext,dtype", [
    (2, 8, 16, 64, 4, torch.bfloat16),     # L - ext >= M: copy from h with an offset
    (3, 12, 10, 64, 3, torch.bfloat16),    # L - ext < M: chains over memory and h
    (2, 5, 9, 6, 2, torch.float32),        # 24-byte rows
    (1, 7, 4, 8, 4, torch.bfloat16),       # ext = L: the memory stays
    (1, 7, 4, 8, 9, torch.bfloat16),       # ext > L: likewise
    (8, 3200, 128, 1024, 64, torch.bfloat16),  # long-memory shape
])
def test_tail_m_ext_len_bit_exact(B, M, L, d, ext, dtype):
    g = torch.Generator().manual_seed(B * 17 + M + L + ext)
    mem = torch.randn(B, M, d, generator=g).to(dtype)
    hid = torch.randn(B, L, d, generator=g).to(dtype)
    expect = oracle.mem_update(bits(mem), bits(hid), M, ext_len=ext)
    dm = mem.cuda()
    txl.mem_update(dm, hid.cuda(), ext_len=ext)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    assert np.array_equal(bits(dm), expect)


@pytest.mark.parametrize("shape,dtype", [
    ((4, 128, 512), torch.bfloat16),          # rows layout [B, M, d]
    ((3, 8, 128, 64), torch.bfloat16),        # heads layout [B, H, M, d_h]
    ((5, 7, 3), torch.float32),               # odd sizes: scalar path
    ((22, 512, 512), torch.bfloat16),         # base-size memory
])
def test_mem_reset_bit_exact(shape, dtype):
    g = torch.Generator().manual_seed(sum(shape))
    mem = torch.randn(*shape, generator=g).to(dtype)
    flags = (torch.arange(shape[0]) % 3 == 1)
    expect = oracle.mem_reset(bits(mem), flags.numpy())
    dm = mem.cuda()
    txl.mem_reset(dm, flags.cuda())
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    assert np.array_equal(bits(dm), expect)
