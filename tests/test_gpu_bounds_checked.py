"""The bounds-checked build (libtxl_checked.so, every computed kernel index
checked, out-of-range accesses skipped and recorded instead of performed)
runs the small parity cases of every entry point: results must match the
oracle as in the plain build and no access may be recorded out of range.

The cases run in a child process with TXL_BOUNDS_CHECKED=1, so that the
binding loads the checked library; this process keeps the plain one."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import oracle
import transformer_xl_relative_attn_gb300 as txl
import txl_workloads as W

assert txl.LIB_PATH.endswith("libtxl_checked.so"), txl.LIB_PATH
assert txl.bounds_status() == (0, 0), "not the bounds-checked build, or stale records"
bf = torch.bfloat16

def tol(r):
    return 1e-2 * float(np.abs(r).max()) + 1e-3

def dev(ci):
    return [t.cuda() for t in (ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb)]

# attention, bf16: ragged query tail, memory not a tile multiple
ci = W.random_call_inputs(1, 2, 200, 136, 64, seed=41)
out = txl.attn_fwd(*dev(ci), scale=ci.scale).float().cpu().double().numpy()
ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)
assert np.abs(out - ref).max() <= tol(ref)
# split-key path through a workspace and through the static scratch
ci = W.random_call_inputs(1, 2, 128, 1500, 64, seed=42)
ws = torch.empty(txl.attn_workspace_bytes(1, 2, 128, 1500, 64), dtype=torch.uint8, device="cuda")
ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)
for o in (txl.attn_fwd_ws(*dev(ci), ws, scale=ci.scale), txl.attn_fwd_noalloc(*dev(ci), scale=ci.scale)):
    assert np.abs(o.float().cpu().double().numpy() - ref).max() <= tol(ref)
# same_length
ci = W.random_call_inputs(1, 2, 256, 256, 64, seed=43)
o = txl.attn_fwd(*dev(ci), ci.scale, same_length=True, mem_len=256).float().cpu().double().numpy()
ref = oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, same_length=True, mem_len=256)
assert np.abs(o - ref).max() <= tol(ref)
# fp32 path
ci = W.random_call_inputs(2, 3, 33, 20, 64, dtype=torch.float32, seed=44)
o = txl.attn_fwd(*dev(ci), scale=ci.scale).cpu().double().numpy()
assert np.abs(o - oracle.attn(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale)).max() <= 1e-5

# memory rolls, bit-exact: L >= M, L < M, ext_len, ring push, reset
g = torch.Generator().manual_seed(5)
def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy()
for (B, M, L, ext) in [(2, 40, 48, 0), (2, 200, 64, 0), (3, 130, 60, 7)]:
    m = torch.randn(B, M, 64, generator=g).to(bf)
    h = torch.randn(B, L, 64, generator=g).to(bf)
    expect = oracle.mem_update(bits(m), bits(h), M, ext_len=ext)
    dm = m.cuda()
    txl.mem_update(dm, h.cuda(), ext_len=ext)
    assert np.array_equal(bits(dm), expect)
ring = torch.randn(2, 256, 64, generator=g).to(bf).cuda()
start = txl.mem_ring_push(ring, torch.randn(2, 64, 64, generator=g).to(bf).cuda(), 224)
assert start == (224 + 64) % 256
flags = torch.tensor([True, False], device="cuda")
txl.mem_reset(ring, flags)
assert float(ring[0].float().abs().sum()) == 0.0 and float(ring[1].float().abs().sum()) > 0

# projections, a Linear with bias / ReLU / residual, a LayerNorm
B, L, M, H = 1, 128, 128, 4
d = H * 64
hx = torch.randn(B, L, d, generator=g).to(bf)
mx = torch.randn(B, M, d, generator=g).to(bf)
w = (torch.randn(3 * d, d, generator=g) * d ** -0.5).to(bf)
q, k, v = txl.qkv_proj(hx.cuda(), mx.cuda(), w.cuda(), H)
for got, r in zip((q, k, v), oracle.qkv_proj(hx, mx, w, H)):
    assert np.abs(got.float().cpu().double().numpy() - r).max() <= tol(r)
wl = (torch.randn(d, d, generator=g) * d ** -0.5).to(bf)
bias = torch.randn(d, generator=g).to(bf)
res = torch.randn(B, L, d, generator=g).to(bf)
y = txl.linear(hx.cuda(), wl.cuda(), bias=bias.cuda(), resid=res.cuda(), relu=True)
ry = np.maximum(oracle.linear(hx.double().numpy(), wl.double().numpy(), bias.double().numpy()), 0) + res.double().numpy()
assert np.abs(y.float().cpu().double().numpy() - ry).max() <= tol(ry)
gam, bet = torch.ones(d).to(bf), torch.zeros(d).to(bf)
ln = txl.layer_norm(hx.cuda(), gam.cuda(), bet.cuda(), y=hx.cuda())
rl = oracle.layer_norm(hx.double().numpy() * 2, gam, bet)
assert np.abs(ln.float().cpu().double().numpy() - rl).max() <= tol(rl)

# backward: fp32 (one row per warp above d_h 64, tiled below), bf16 on the
# CUDA cores and on the tensor cores (several query and key tiles, ragged),
# and the tensor-core backward from the forward's saved out and lse
cases = [(torch.float32, 32, 40, 24, 1e-4, 1e-5, "cc"), (torch.float32, 128, 40, 24, 1e-4, 1e-5, "cc"),
         (bf, 64, 40, 24, 1e-2, 1e-3, "cc"), (bf, 64, 200, 100, 1e-2, 1e-3, "tc"),
         (bf, 64, 200, 100, 1e-2, 1e-3, "saved")]
for dt, dh, Lq, Mq, rt, at, path in cases:
    ci = W.random_call_inputs(1, 2, Lq, Mq, dh, dtype=dt, std=0.5, seed=dh + Lq)
    gout = torch.randn(1, 2, Lq, dh, generator=g).to(dt)
    if path == "saved":
        o_s, lse_s = txl.attn_fwd_lse(*dev(ci), scale=ci.scale)
        got = txl.attn_bwd(*dev(ci), gout.cuda(), ci.scale, out=o_s, lse=lse_s)
    else:
        got = txl.attn_bwd(*dev(ci), gout.cuda(), ci.scale, tensor_cores=(path == "tc"))
    ref = oracle.attn_bwd(ci.q, ci.k, ci.v, ci.r_k, ci.u, ci.vb, ci.scale, gout)
    for n in ("dq", "dk", "dv", "dr", "du", "dvb"):
        r = ref[n]
        assert np.abs(got[n].cpu().double().numpy() - r).max() <= rt * np.abs(r).max() + at, (path, n)

torch.cuda.synchronize()
assert txl.sync_status() == 0
st, first = txl.bounds_status()
assert (st, first) == (0, 0), f"bounds violation recorded: status {st}, record {first:#x}"
print("bounds-checked build: all cases in range and at parity")
'''


def test_bounds_checked_build_runs_every_entry_point_in_range():
    lib = os.path.join(ROOT, "transformer_xl_relative_attn_gb300", "libtxl_checked.so")
    assert os.path.exists(lib), "libtxl_checked.so missing: run __graft_entry__.build()"
    env = dict(os.environ, TXL_BOUNDS_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "all cases in range" in r.stdout
