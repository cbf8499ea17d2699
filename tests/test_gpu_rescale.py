"""The online softmax's rescale of the running output, forced on the GPU.

The pages' softmax runs over all of a query's visible keys
("Transformer-XL模型 核心源码阅读笔记", RelPartialLearnableMultiHeadAttn.forward:
softmax over the key axis of AC + BD; "Transformer-XL" notes, section
"Relative Positional Encoding": the score inside that softmax).  A kernel that
sweeps the keys tile by tile keeps a running maximum and must scale what it
has accumulated whenever a later tile raises that maximum.  The bf16 kernel
does so only when a tile's maximum exceeds the running one by more than 8
log2 units, and then with a factor 0 < alpha < 1 on O in tensor memory.

Random inputs almost never trigger that: their scores spread over a few log2
units.  Here the content term climbs in a staircase along the keys: q has a
unit component on axis 0 and k_j carries c * j / 64 there, so each 64-key
tile's scores sit about ``STEP`` log2 units above the previous tile's (and
2 * STEP above the previous tile of the same softmax group).  Every row
therefore rescales several times, with alpha = 2^-(jump) strictly between 0
and 1, in both key-tile groups.  Small random terms on the other axes keep
each tile's distribution non-degenerate.  The output is compared element by
element with the fp64 oracle at the bf16 tolerance (1e-2 * max|ref| + 1e-3);
the fp32 path's per-chunk rescale gets a twin at 1e-5.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

pytestmark = pytest.mark.gpu

STEP = 10.0       # log2 units gained per 64 keys by the staircase
LOG2E = 1.0 / math.log(2.0)


def staircase_inputs(B, H, L, M, dh=64, dtype=torch.bfloat16, seed=0, step=STEP, scale=0.125,
                     per=64.0):
    """Inputs whose content scores rise by ``step`` log2 units every ``per``
    keys (a continuous ramp: each tile's own maximum also climbs)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    K = M + L

    def n(*shape, s):
        return torch.empty(shape, dtype=torch.float32).normal_(0.0, s, generator=g)

    q = n(B, H, L, dh, s=0.3)
    q[..., 0] = 1.0
    k = n(B, H, K, dh, s=0.3)
    slope = step / (scale * LOG2E) / per          # natural-log units of q.k per key
    k[..., 0] = slope * torch.arange(K, dtype=torch.float32) + n(B, H, K, s=0.2)
    v = n(B, H, K, dh, s=1.0)
    r = n(K, H, dh, s=0.3)
    u = n(H, dh, s=0.1)
    u[:, 0] = 0.0                                  # keep the slope exactly c
    vb = n(H, dh, s=0.1)
    c = [t.to(dtype) for t in (q, k, v, r, u, vb)]
    return W.CallInputs(*c, scale)


def max_jumps_log2(ci, row_pairs=4):
    """Largest rises of the running maximum between consecutive 64-key tiles
    of the same parity (each group's view), over a few rows: the test inputs'
    own property that the rescale must fire (computed here from the inputs,
    in fp64, only to document the case)."""
    q, k, r, u, vb = (t.double() for t in (ci.q, ci.k, ci.r_k, ci.u, ci.vb))
    B, H, L, dh = q.shape
    K = k.shape[2]
    M = K - L
    jumps = []
    for p in range(min(row_pairs, B * H)):
        b, h = divmod(p, H)
        for i in (0, L // 2, L - 1):
            j = torch.arange(M + i + 1)
            ac = (q[b, h, i] + u[h]) @ k[b, h, j].T
            bd = (q[b, h, i] + vb[h]) @ r[K - 1 - (M + i - j), h].T
            s = (ci.scale * (ac + bd) * LOG2E).numpy()
            tiles = [s[t * 64:(t + 1) * 64].max() for t in range((M + i) // 64 + 1)]
            for g in (0, 1):
                mx = -np.inf
                for t in range(g, len(tiles), 2):
                    if mx > -np.inf:
                        jumps.append(tiles[t] - mx)
                    mx = max(mx, tiles[t])
    return np.array(jumps)


def bf16_check(got, ci, same_length=False, mem_len=None):
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, same_length=same_length,
                      mem_len=mem_len)
    got = got.float().cpu().double().numpy()
    assert np.isfinite(got).all()
    tol = 1e-2 * np.abs(ref).max() + 1e-3
    err = np.abs(got - ref).max()
    assert err <= tol, f"max|d| = {err}, tol = {tol}"


def dev(ci):
    return [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]


@pytest.mark.parametrize("B,H,L,M", [
    (1, 2, 200, 0),       # no memory, ragged query tail: climbs across the diagonal tiles
    (2, 2, 128, 136),     # memory not a tile multiple
    (1, 3, 130, 1000),    # long memory: many rescales per row
    (2, 1, 384, 512),     # several query tiles per (b, h)
])
def test_bf16_rescale_fires_and_matches_oracle(B, H, L, M):
    ci = staircase_inputs(B, H, L, M, seed=B * 31 + L + M)
    j = max_jumps_log2(ci)
    # every group's tile maximum rises past the 8-unit threshold, so the
    # kernel rescales O with 0 < alpha < 1 (not the alpha = 0 first tile)
    assert (j > 8.0).mean() > 0.9 and np.isfinite(j).all()
    out = txl.attn_fwd(*dev(ci), scale=ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    bf16_check(out, ci)


@pytest.mark.parametrize("B,H,L,M", [(1, 2, 128, 3000), (2, 2, 200, 1500)])
def test_bf16_rescale_on_split_key_path(B, H, L, M):
    """The workspace entry point splits each item's keys over several units;
    every unit rescales within its share and the combine pass merges them."""
    ci = staircase_inputs(B, H, L, M, seed=M, step=9.0)
    need = txl.attn_workspace_bytes(B, H, L, M, 64)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = txl.attn_fwd_ws(*dev(ci), ws, scale=ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    bf16_check(out, ci)


@pytest.mark.parametrize("B,H,L,M,mem_len", [(1, 2, 256, 256, 256), (2, 1, 512, 512, 512)])
def test_bf16_rescale_same_length(B, H, L, M, mem_len):
    """same_length: a row's first processed tiles are wholly below its lower
    key bound (masked), then the first visible tile, then the climb."""
    ci = staircase_inputs(B, H, L, M, seed=L + 7)
    out = txl.attn_fwd(*dev(ci), scale=ci.scale, same_length=True, mem_len=mem_len)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    bf16_check(out, ci, same_length=True, mem_len=mem_len)


@pytest.mark.parametrize("L,M", [(40, 60), (33, 70)])
def test_f32_rescale_matches_oracle(L, M):
    """fp32 path (32-key chunks, a rescale on every chunk whose maximum is
    higher): a gentler climb over few keys, so that the fp32 rounding of the
    large scores stays well below 1e-5."""
    ci = staircase_inputs(1, 2, L, M, dh=64, dtype=torch.float32, seed=L, step=4.0, per=32.0)
    out = txl.attn_fwd(*dev(ci), scale=ci.scale)
    torch.cuda.synchronize()
    assert txl.sync_status() == 0
    ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)
    assert np.abs(out.cpu().double().numpy() - ref).max() <= 1e-5
