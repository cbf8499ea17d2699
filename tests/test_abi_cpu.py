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
