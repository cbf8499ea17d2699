"""Host-side checks of libtxl.so that need no GPU: the library loads, exports
every function include/txl_attn.h declares, and rejects bad arguments before
anything is launched."""
import ctypes
import subprocess

import pytest

import transformer_xl_relative_attn_gb300 as txl
from transformer_xl_relative_attn_gb300 import _lib

A = 0x10000  # a fake, 16-byte aligned, never dereferenced device address


@pytest.fixture(scope="module")
def lib():
    return txl.load()


def test_header_declares_the_contract():
    names = set(txl.header_functions())
    assert {"txl_attn_fwd", "txl_mem_update", "txl_attn_fwd_ws", "txl_attn_workspace_bytes",
            "txl_sync_status", "txl_status_string", "txl_version", "txl_debug_inject"} <= names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", txl.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for name in txl.header_functions():
        assert name in exported, name
        getattr(lib, name)


def test_status_strings_and_version(lib):
    for code, name in _lib.STATUS.items():
        assert txl.status_string(code)
    assert txl.status_string(-6) == "device-side wait timed out"
    assert txl.version() == (1, 0)


def call_attn(lib, q=A, k=A, v=A, r=A, u=A, vb=A, B=1, H=1, L=4, M=3, dh=64, out=A + (1 << 30),
              dtype=txl.TXL_BF16):
    return lib.txl_attn_fwd(q, k, v, r, u, vb, B, H, L, M, dh, 0.125, out, dtype, None)


def test_attn_rejects_bad_arguments(lib):
    assert call_attn(lib, q=None) == -1
    assert call_attn(lib, out=None) == -1
    assert call_attn(lib, B=0) == -1
    assert call_attn(lib, L=0) == -1
    assert call_attn(lib, M=-1) == -1
    assert call_attn(lib, dtype=7) == -1
    assert call_attn(lib, dh=32) == -2           # bf16 path is d_h = 64 only
    assert call_attn(lib, dh=512, dtype=txl.TXL_F32) == -2
    assert call_attn(lib, q=A + 8) == -3         # misaligned
    assert call_attn(lib, out=A + 4) == -3
    assert call_attn(lib, out=A) == -4           # output aliases the inputs


def test_ws_and_workspace_query(lib):
    assert lib.txl_attn_workspace_bytes(0, 1, 1, 1, 64, 1) == 0
    assert lib.txl_attn_fwd_ws(None, A, A, A, A, A, 1, 1, 4, 3, 64, 0.1, A + (1 << 30), 1,
                               None, 0, None) == -1


def test_mem_update_validation(lib):
    assert lib.txl_mem_update(A, A + (1 << 30), 2, 4, 0, 8, txl.TXL_BF16, None) == 0  # M = 0: no-op
    assert lib.txl_mem_update(None, A, 2, 4, 3, 8, txl.TXL_BF16, None) == -1
    assert lib.txl_mem_update(A, A, 2, 4, 3, 8, 9, None) == -1
    assert lib.txl_mem_update(A, A + 16, 2, 4, 3, 8, txl.TXL_BF16, None) == -4       # overlap


def test_debug_inject_validation(lib):
    assert lib.txl_debug_inject(5) == -1
    assert lib.txl_debug_inject(0) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 7, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        txl.attn_fwd(q, k, k, torch.zeros(7, 1, 64, dtype=torch.bfloat16),
                     torch.zeros(1, 64, dtype=torch.bfloat16), torch.zeros(1, 64, dtype=torch.bfloat16))


def test_binding_refuses_tensors_on_another_device():
    """Every tensor of a call must be on the first tensor's device: the C call
    runs with that device current, and a pointer from another device would be
    dereferenced on the wrong GPU.  (On this CPU-only host the check is
    exercised directly: a tensor whose device differs from the call's.)"""
    import torch
    other = torch.device("cuda", 1)
    with pytest.raises(ValueError, match="cuda:1"):
        _lib._need(torch.zeros(2, 64), "k", (2, 64), torch.float32, other)
    with pytest.raises(ValueError, match="on cpu"):
        _lib._need(torch.zeros(2, 64), "k", (2, 64), torch.float32, other)


def test_status_table_covers_every_header_code():
    """Each TXL_ERR_* code the header defines has a name in the binding."""
    import re
    with open(_lib.HEADER, encoding="utf-8") as fh:
        codes = {int(v) for v in re.findall(r"\bTXL_(?:OK|ERR_\w+)\s*=\s*(-?\d+)", fh.read())}
    assert codes and codes <= set(_lib.STATUS)


# --------------------------------------------------------------------------
# the entry points added beyond the attention operator: bad arguments are
# rejected on the host, before any CUDA call
# --------------------------------------------------------------------------
O = A + (1 << 30)   # a second fake address, far from A


def test_attn_fwd_ex_rejects_bad_mem_len(lib):
    def call(**kw):
        a = dict(same_length=1, mem_len=3)
        a.update(kw)
        return lib.txl_attn_fwd_ex(A, A, A, A, A, A, 1, 1, 4, 3, 64, 0.125, a["same_length"], a["mem_len"],
                                   O, txl.TXL_BF16, None)
    assert call(mem_len=2) == -1      # mem_len < M
    assert call(mem_len=-1) == -1


def test_qkv_proj_rejects_bad_sizes_layouts_and_rings(lib):
    def call(h_layout=0, mem_layout=0, start=0, L=128, M=128, H=4, dh=64, q=O, k=O + (1 << 26), v=O + (1 << 27)):
        return lib.txl_qkv_proj_ring(A, h_layout, A + (1 << 24), mem_layout, start, A + (1 << 25), 1, L, M, H,
                                     dh, q, k, v, None)
    assert call(h_layout=2) == -1
    assert call(mem_layout=-1) == -1
    assert call(start=128) == -1      # start must be < M
    assert call(start=64, M=256) == -2  # not a multiple of 128
    assert call(L=100) == -2
    assert call(dh=32) == -2
    assert call(H=6) == -2
    assert call(q=O + 8) == -3
    assert call(q=A) == -4            # q over h


def test_linear_and_layer_norm_reject_bad_arguments(lib):
    def lin(x_layout=0, T=128, K=256, N=256, out=O, resid=0, bias=0):
        return lib.txl_linear(A, x_layout, 1, T, K, A + (1 << 25), N, bias, resid, 0, out, None)
    assert lin(x_layout=3) == -1
    assert lin(T=100) == -2
    assert lin(K=100) == -2
    assert lin(N=128) == -2
    assert lin(out=O + 2) == -3
    assert lin(out=A) == -4
    assert lin(resid=O + 64) == -4    # partly overlapping the output
    def ln(d=512, out=O, y=0, eps=1e-5):
        return lib.txl_layer_norm(A, y, A + (1 << 25), A + (1 << 26), 64, d, ctypes.c_float(eps), out, None)
    assert ln(d=500) == -2
    assert ln(d=1280) == -2
    assert ln(eps=-1.0) == -1
    assert ln(out=O + 4) == -3
    assert ln(out=A + 64) == -4       # overlaps x without being x


def test_memory_calls_reject_bad_arguments(lib):
    new = ctypes.c_int(-1)
    assert lib.txl_mem_update_ext(A, O, 1, 4, 3, 8, -1, txl.TXL_BF16, None) == -1
    assert lib.txl_mem_ring_push(A, O, 1, 4, 8, 8, 8, ctypes.byref(new), txl.TXL_BF16, None) == -1  # start >= M
    assert lib.txl_mem_ring_push(A, O, 1, 4, 8, 8, 0, None, txl.TXL_BF16, None) == -1
    assert lib.txl_mem_ring_push(A, A + 16, 1, 4, 8, 8, 0, ctypes.byref(new), txl.TXL_BF16, None) == -4
    assert lib.txl_mem_reset(A, 0, 2, 8, 8, txl.TXL_BF16, None) == -1   # no flags
    assert lib.txl_mem_reset(A, A + 16, 2, 8, 8, txl.TXL_BF16, None) == -4


def test_attn_bwd_rejects_bad_arguments(lib):
    g = [O + (i << 24) for i in range(6)]
    def call(dh=64, dtype=txl.TXL_BF16, grads=g, same_length=0, mem_len=3):
        return lib.txl_attn_bwd(A, A, A, A, A, A, A, 1, 1, 4, 3, dh, 0.125, same_length, mem_len, *grads,
                                dtype, None)
    assert call(dtype=5) == -1
    assert call(dh=512) == -2
    assert call(grads=[O + 4] + g[1:]) == -3
    assert call(grads=[A] + g[1:]) == -4           # dq over the inputs
    assert call(grads=[g[0], g[0]] + g[2:]) == -4  # two gradients overlap
    assert call(same_length=1, mem_len=1) == -1


def test_plain_build_reports_no_bounds_checks(lib):
    """txl_bounds_status is a bounds-checked-build facility: the plain library
    answers TXL_ERR_UNSUPPORTED without touching the GPU."""
    st, first = txl.bounds_status()
    assert st == -2 and first == 0


def test_checked_build_exports_the_same_symbols():
    """libtxl_checked.so (the -DTXL_CHECKED build of the same sources) exports
    every function the header declares, like libtxl.so."""
    import os
    path = os.path.join(os.path.dirname(txl.LIB_PATH), "libtxl_checked.so")
    assert os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    assert set(txl.header_functions()) <= exported


def test_qkvr_proj_rejects_bad_arguments(lib):
    """txl_qkvr_proj: the q/k/v contract, the r_proj contract over M+L rows,
    and no overlap between r_k and the other arguments."""
    X = A + (1 << 32)

    def call(**kw):
        a = dict(h=A, mem=A + (1 << 28), w=A + (2 << 28), emb=A + (3 << 28), wr=A + (4 << 28), B=1, L=128,
                 M=128, H=4, dh=64, q=O, k=O + (1 << 28), v=O + (2 << 28), r=X)
        a.update(kw)
        return lib.txl_qkvr_proj(a["h"], 0, a["mem"], 0, 0, a["w"], a["emb"], a["wr"], a["B"], a["L"], a["M"],
                                 a["H"], a["dh"], a["q"], a["k"], a["v"], a["r"], None)
    assert call(emb=None) == -1
    assert call(r=None) == -1
    assert call(L=100) == -2             # not a multiple of 128
    assert call(dh=32) == -2
    assert call(emb=A + (3 << 28) + 8) == -3
    assert call(r=O) == -4               # r_k overlaps q
    assert call(r=A) == -4               # r_k overlaps h
