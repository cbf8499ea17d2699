"""ctypes binding of libtxl.so (include/txl_attn.h).  Argument marshalling only:
every step of the computation runs in the library's CUDA kernels.  There is
no CPU fallback: if the library is missing, every call raises."""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
# TXL_BOUNDS_CHECKED=1 selects the bounds-checked build of the same library
LIB_PATH = os.path.join(PKG, "libtxl_checked.so" if os.environ.get("TXL_BOUNDS_CHECKED") == "1"
                        else "libtxl.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "txl_attn.h")

TXL_F32 = 0
TXL_BF16 = 1

STATUS = {
    0: "TXL_OK",
    -1: "TXL_ERR_INVALID_ARG",
    -2: "TXL_ERR_UNSUPPORTED",
    -3: "TXL_ERR_MISALIGNED",
    -4: "TXL_ERR_ALIAS",
    -5: "TXL_ERR_LAUNCH",
    -6: "TXL_ERR_DEVICE_TIMEOUT",
    -7: "TXL_ERR_WORKSPACE",
    -8: "TXL_ERR_CUDA",
    -9: "TXL_ERR_SCRATCH_LIMIT",
    -10: "TXL_ERR_OUT_OF_BOUNDS",
}

_lib = None
_lock = threading.Lock()


class TxlError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        name = STATUS.get(code, str(code))
        super().__init__(f"{what}: {name} ({status_string(code)})")


def load() -> ctypes.CDLL:
    """Loads libtxl.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(the CUDA library is required; there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.txl_attn_fwd.argtypes = [vp] * 6 + [i] * 5 + [f, vp, i, vp]
        lib.txl_attn_fwd.restype = i
        lib.txl_attn_fwd_ex.argtypes = [vp] * 6 + [i] * 5 + [f, i, i, vp, i, vp]
        lib.txl_attn_fwd_ex.restype = i
        lib.txl_attn_bwd.argtypes = [vp] * 7 + [i] * 5 + [f, i, i] + [vp] * 6 + [i, vp]
        lib.txl_attn_bwd.restype = i
        lib.txl_attn_bwd_workspace_bytes.argtypes = [i] * 7
        lib.txl_attn_bwd_workspace_bytes.restype = sz
        lib.txl_attn_bwd_ws.argtypes = [vp] * 7 + [i] * 5 + [f, i, i] + [vp] * 6 + [i, vp, sz, vp]
        lib.txl_attn_bwd_ws.restype = i
        lib.txl_attn_fwd_lse.argtypes = [vp] * 6 + [i] * 5 + [f, vp, vp, i, vp]
        lib.txl_attn_fwd_lse.restype = i
        lib.txl_attn_bwd_saved.argtypes = [vp] * 9 + [i] * 5 + [f] + [vp] * 6 + [i, vp, sz, vp]
        lib.txl_attn_bwd_saved.restype = i
        lib.txl_attn_fwd_ws.argtypes = [vp] * 6 + [i] * 5 + [f, vp, i, vp, sz, vp]
        lib.txl_attn_fwd_ws.restype = i
        lib.txl_attn_fwd_noalloc.argtypes = [vp] * 6 + [i] * 5 + [f, vp, i, vp]
        lib.txl_attn_fwd_noalloc.restype = i
        lib.txl_qkv_proj.argtypes = [vp] * 3 + [i] * 5 + [vp] * 4
        lib.txl_qkv_proj.restype = i
        lib.txl_qkv_proj_ex.argtypes = [vp, i, vp, i, vp] + [i] * 5 + [vp] * 4
        lib.txl_qkv_proj_ex.restype = i
        lib.txl_qkv_proj_ring.argtypes = [vp, i, vp, i, i, vp] + [i] * 5 + [vp] * 4
        lib.txl_qkv_proj_ring.restype = i
        lib.txl_mem_ring_push.argtypes = [vp, vp] + [i] * 5 + [ctypes.POINTER(ctypes.c_int), i, vp]
        lib.txl_mem_ring_push.restype = i
        lib.txl_qkvr_proj.argtypes = [vp, i, vp, i, i, vp, vp, vp] + [i] * 5 + [vp] * 5
        lib.txl_qkvr_proj.restype = i
        lib.txl_r_proj.argtypes = [vp, vp] + [i] * 3 + [vp, vp]
        lib.txl_r_proj.restype = i
        lib.txl_attn_workspace_bytes.argtypes = [i] * 6
        lib.txl_attn_workspace_bytes.restype = sz
        lib.txl_mem_update.argtypes = [vp, vp] + [i] * 5 + [vp]
        lib.txl_mem_update.restype = i
        lib.txl_linear.argtypes = [vp, i, i, i, i, vp, i, vp, vp, i, vp, vp]
        lib.txl_linear.restype = i
        lib.txl_layer_norm.argtypes = [vp, vp, vp, vp, ctypes.c_longlong, i, f, vp, vp]
        lib.txl_layer_norm.restype = i
        lib.txl_mem_update_ext.argtypes = [vp, vp] + [i] * 6 + [vp]
        lib.txl_mem_update_ext.restype = i
        lib.txl_mem_reset.argtypes = [vp, vp] + [i] * 4 + [vp]
        lib.txl_mem_reset.restype = i
        lib.txl_sync_status.argtypes = [vp]
        lib.txl_sync_status.restype = i
        lib.txl_status_string.argtypes = [i]
        lib.txl_status_string.restype = ctypes.c_char_p
        lib.txl_version.argtypes = []
        lib.txl_version.restype = i
        lib.txl_debug_inject.argtypes = [i]
        lib.txl_debug_inject.restype = i
        lib.txl_bounds_status.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
        lib.txl_bounds_status.restype = i
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions include/txl_attn.h declares."""
    with open(HEADER, encoding="utf-8") as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(txl_\w+)\s*\(", text, flags=re.M)


def status_string(code: int) -> str:
    return load().txl_status_string(int(code)).decode()


def version() -> tuple[int, int]:
    v = load().txl_version()
    return v >> 16, v & 0xFFFF


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TXL_BF16
    if t.dtype == torch.float32:
        return TXL_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32 only")


def _invoke(device, name: str, *args):
    """Calls C entry point ``name`` with ``device`` current, so that the
    library's launches, its status word and its static scratch are those of
    the device the call's tensors live on."""
    with torch.cuda.device(device):
        return getattr(load(), name)(*args)


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, shape: tuple, dtype, device=None) -> None:
    """Type, device, dtype, shape and contiguity of one argument.  ``device``:
    the device every tensor of the call must share (the kernels run there)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's other tensors on {device}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _attn_args(q, k, v, r_k, u, vb, scale, out):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d_h]")
    B, H, L, dh = q.shape
    K = k.shape[2] if k.dim() == 4 else -1
    M = K - L
    if M < 0:
        raise ValueError("k must be [B, H, M+L, d_h] with M >= 0")
    dt = q.dtype
    _need(q, "q", (B, H, L, dh), dt)
    dv = q.device
    _need(k, "k", (B, H, K, dh), dt, dv)
    _need(v, "v", (B, H, K, dh), dt, dv)
    _need(r_k, "r_k", (K, H, dh), dt, dv)
    _need(u, "u", (H, dh), dt, dv)
    _need(vb, "v_bias", (H, dh), dt, dv)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (B, H, L, dh), dt, dv)
    if scale is None:
        scale = dh ** -0.5
    return B, H, L, M, dh, float(scale), out


def attn_fwd(q, k, v, r_k, u, vb, scale=None, out=None, stream=None, same_length=False,
             mem_len=None) -> torch.Tensor:
    """Relative attention forward (txl_attn_fwd, or txl_attn_fwd_ex with
    same_length).  Shapes: q [B,H,L,dh]; k, v [B,H,M+L,dh] (memory rows
    first); r_k [M+L,H,dh] (row r <-> distance M+L-1-r); u, vb [H,dh].
    same_length: every query attends over the same number of keys, for the
    configured memory length mem_len (default M).  Returns out [B,H,L,dh]."""
    B, H, L, M, dh, scale, out = _attn_args(q, k, v, r_k, u, vb, scale, out)
    if same_length:
        rc = _invoke(q.device, "txl_attn_fwd_ex", q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(),
                                    u.data_ptr(), vb.data_ptr(), B, H, L, M, dh, scale, 1,
                                    M if mem_len is None else int(mem_len), out.data_ptr(),
                                    _dtype_code(q), _stream(stream, q.device))
        if rc != 0:
            raise TxlError(rc, "txl_attn_fwd_ex")
        return out
    rc = _invoke(q.device, "txl_attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(),
                             u.data_ptr(), vb.data_ptr(), B, H, L, M, dh, scale, out.data_ptr(),
                             _dtype_code(q), _stream(stream, q.device))
    if rc != 0:
        raise TxlError(rc, "txl_attn_fwd")
    return out


def attn_bwd_workspace_bytes(B, H, L, M, dh, dtype=torch.bfloat16, same_length=False, device=None) -> int:
    """txl_attn_bwd_workspace_bytes: scratch of the tensor-core backward (0
    when the call takes the CUDA-core path)."""
    code = TXL_BF16 if dtype == torch.bfloat16 else TXL_F32
    dev = device if device is not None else torch.cuda.current_device()
    return int(_invoke(dev, "txl_attn_bwd_workspace_bytes", B, H, L, M, dh, code, int(bool(same_length))))


def attn_fwd_lse(q, k, v, r_k, u, vb, scale=None, out=None, lse=None, stream=None):
    """txl_attn_fwd_lse: attn_fwd (bf16, d_h = 64) that also returns each query
    row's log2-sum-exp of its scores, lse [B, H, L] fp32: (out, lse)."""
    B, H, L, M, dh, scale, out = _attn_args(q, k, v, r_k, u, vb, scale, out)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need(lse, "lse", (B, H, L), torch.float32, q.device)
    rc = _invoke(q.device, "txl_attn_fwd_lse", q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(),
                 u.data_ptr(), vb.data_ptr(), B, H, L, M, dh, scale, out.data_ptr(), lse.data_ptr(), _dtype_code(q),
                 _stream(stream, q.device))
    if rc != 0:
        raise TxlError(rc, "txl_attn_fwd_lse")
    return out, lse


def attn_bwd(q, k, v, r_k, u, vb, dout, scale=None, same_length=False, mem_len=None, stream=None,
             tensor_cores=True, workspace=None, grads=None, out=None, lse=None):
    """fp32 gradients of sum(out * dout) with respect to q, k, v, r_k, u and
    vb (stop-gradient memory: the memory rows' dk, dv are included and left
    to the caller).  Returns a dict dq, dk, dv, dr, du, dvb.

    tensor_cores: txl_attn_bwd_ws (the tcgen05 passes where they apply: bf16,
    d_h = 64, no same_length; otherwise the same as txl_attn_bwd); False:
    txl_attn_bwd, the CUDA-core kernels.  workspace: a uint8 tensor on the
    device of at least attn_bwd_workspace_bytes(...) bytes (allocated here
    when None); grads: a dict of preallocated gradient tensors to fill.
    out, lse: the forward's saved output and row log2-sum-exp (attn_fwd_lse):
    txl_attn_bwd_saved, which takes them instead of recomputing the forward."""
    B, H, L, M, dh, scale, _ = _attn_args(q, k, v, r_k, u, vb, scale, dout)
    _need(dout, "dout", (B, H, L, dh), q.dtype, q.device)
    f32 = dict(dtype=torch.float32, device=q.device)
    shapes = {"dq": (B, H, L, dh), "dk": (B, H, M + L, dh), "dv": (B, H, M + L, dh), "dr": (M + L, H, dh),
              "du": (H, dh), "dvb": (H, dh)}
    if grads is None:
        g = {n: torch.empty(sh, **f32) for n, sh in shapes.items()}
    else:
        g = grads
        for n, sh in shapes.items():
            _need(g[n], n, sh, torch.float32, q.device)
    ml = M if mem_len is None else int(mem_len)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(), u.data_ptr(), vb.data_ptr(), dout.data_ptr(),
            B, H, L, M, dh, scale, int(bool(same_length)), ml,
            *[g[n].data_ptr() for n in ("dq", "dk", "dv", "dr", "du", "dvb")], _dtype_code(q))
    if (out is None) != (lse is None):
        raise ValueError("out and lse are given together")
    if out is not None:
        _need(out, "out", (B, H, L, dh), q.dtype, q.device)
        _need(lse, "lse", (B, H, L), torch.float32, q.device)
        need = attn_bwd_workspace_bytes(B, H, L, M, dh, q.dtype, False, q.device)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        rc = _invoke(q.device, "txl_attn_bwd_saved", q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(),
                     u.data_ptr(), vb.data_ptr(), out.data_ptr(), lse.data_ptr(), dout.data_ptr(), B, H, L, M, dh,
                     scale, *[g[n].data_ptr() for n in ("dq", "dk", "dv", "dr", "du", "dvb")], _dtype_code(q),
                     workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream, q.device))
        if rc != 0:
            raise TxlError(rc, "txl_attn_bwd_saved")
        return g
    if tensor_cores:
        need = attn_bwd_workspace_bytes(B, H, L, M, dh, q.dtype, same_length, q.device)
        if workspace is None and need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None and (not isinstance(workspace, torch.Tensor) or workspace.device != q.device):
            raise ValueError(f"workspace must be a tensor on {q.device}")
        wp = workspace.data_ptr() if workspace is not None else 0
        wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = _invoke(q.device, "txl_attn_bwd_ws", *args, wp, wn, _stream(stream, q.device))
        name = "txl_attn_bwd_ws"
    else:
        rc = _invoke(q.device, "txl_attn_bwd", *args, _stream(stream, q.device))
        name = "txl_attn_bwd"
    if rc != 0:
        raise TxlError(rc, name)
    return g


def attn_workspace_bytes(B, H, L, M, dh, dtype=torch.bfloat16, device=None) -> int:
    """txl_attn_workspace_bytes for a call on ``device`` (default: the current
    one): the split depends on that device's SM count."""
    code = TXL_BF16 if dtype == torch.bfloat16 else TXL_F32
    dev = device if device is not None else torch.cuda.current_device()
    return int(_invoke(dev, "txl_attn_workspace_bytes", B, H, L, M, dh, code))


def attn_fwd_ws(q, k, v, r_k, u, vb, workspace, scale=None, out=None, stream=None):
    """txl_attn_fwd_ws: like attn_fwd with caller-owned scratch (a uint8 CUDA
    tensor of at least attn_workspace_bytes(...) bytes, or None when 0)."""
    B, H, L, M, dh, scale, out = _attn_args(q, k, v, r_k, u, vb, scale, out)
    if workspace is not None and (not isinstance(workspace, torch.Tensor) or workspace.device != q.device):
        raise ValueError(f"workspace must be a tensor on {q.device}")
    wp = workspace.data_ptr() if workspace is not None else 0
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _invoke(q.device, "txl_attn_fwd_ws", q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(),
                                u.data_ptr(), vb.data_ptr(), B, H, L, M, dh, scale, out.data_ptr(),
                                _dtype_code(q), wp, wn, _stream(stream, q.device))
    if rc != 0:
        raise TxlError(rc, "txl_attn_fwd_ws")
    return out


def attn_fwd_noalloc(q, k, v, r_k, u, vb, scale=None, out=None, stream=None):
    """txl_attn_fwd_noalloc: like attn_fwd_ws, with the library's static
    device scratch instead of a caller workspace (calls on one device must not
    overlap in time; the first call on a device must not be captured)."""
    B, H, L, M, dh, scale, out = _attn_args(q, k, v, r_k, u, vb, scale, out)
    rc = _invoke(q.device, "txl_attn_fwd_noalloc", q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(),
                                     u.data_ptr(), vb.data_ptr(), B, H, L, M, dh, scale,
                                     out.data_ptr(), _dtype_code(q), _stream(stream, q.device))
    if rc != 0:
        raise TxlError(rc, "txl_attn_fwd_noalloc")
    return out


def _qkv_args(h, mem, w_qkv, H, q, k, v):
    """Shapes, layouts and outputs of the q/k/v projections (txl_qkv_proj_ex's
    contract); returns (q, k, v, (B, L, M))."""
    if h.dim() == 3:
        B, L, d = h.shape
        h_layout = 0
    elif h.dim() == 4:
        B, Hh, L, dh_ = h.shape
        if Hh != H:
            raise ValueError("h in the heads layout must have H heads")
        d = H * dh_
        h_layout = 1
    else:
        raise ValueError("h must be [B, L, d] or [B, H, L, d_h]")
    dh = d // H
    if mem.dim() == 3:
        M = mem.shape[1]
        mem_shape = (B, M, d)
    elif mem.dim() == 4:
        M = mem.shape[2]
        mem_shape = (B, H, M, dh)
    else:
        raise ValueError("mem must be [B, M, d] or [B, H, M, d_h]")
    _need(h, "h", (B, L, d) if h_layout == 0 else (B, H, L, dh), torch.bfloat16)
    if M > 0:
        _need(mem, "mem", mem_shape, torch.bfloat16, h.device)
    _need(w_qkv, "w_qkv", (3 * d, d), torch.bfloat16, h.device)
    if q is None:
        q = torch.empty((B, H, L, dh), dtype=torch.bfloat16, device=h.device)
    if k is None:
        k = torch.empty((B, H, M + L, dh), dtype=torch.bfloat16, device=h.device)
    if v is None:
        v = torch.empty((B, H, M + L, dh), dtype=torch.bfloat16, device=h.device)
    _need(q, "q", (B, H, L, dh), torch.bfloat16, h.device)
    _need(k, "k", (B, H, M + L, dh), torch.bfloat16, h.device)
    _need(v, "v", (B, H, M + L, dh), torch.bfloat16, h.device)
    return q, k, v, (B, L, M)


def qkv_proj(h, mem, w_qkv, H, q=None, k=None, v=None, stream=None, mem_start=0):
    """txl_qkv_proj_ex: q = h W_q^T, k/v = [mem; h] W_{k,v}^T split into heads.
    h is [B, L, d] (rows) or [B, H, L, d_h] (heads: an attention output),
    mem likewise [B, M, d] or [B, H, M, d_h] (M may be 0); w_qkv [3d, d]; bf16
    CUDA tensors.  mem_start: mem is a ring whose logical row 0 is stored at
    row mem_start (txl_qkv_proj_ring).  Returns (q [B, H, L, d_h], k, v
    [B, H, M+L, d_h])."""
    q, k, v, (B, L, M) = _qkv_args(h, mem, w_qkv, H, q, k, v)
    dh = q.shape[3]
    h_layout = 0 if h.dim() == 3 else 1
    mem_layout = 0 if mem.dim() == 3 else 1
    rc = _invoke(h.device, "txl_qkv_proj_ring", h.data_ptr(), h_layout, mem.data_ptr() if M > 0 else 0,
                 mem_layout, int(mem_start), w_qkv.data_ptr(), B, L, M, H, dh, q.data_ptr(),
                 k.data_ptr(), v.data_ptr(), _stream(stream, h.device))
    if rc != 0:
        raise TxlError(rc, "txl_qkv_proj_ring")
    return q, k, v


def qkvr_proj(h, mem, w_qkv, emb, w_r, H, q=None, k=None, v=None, r_k=None, stream=None, mem_start=0):
    """txl_qkvr_proj: qkv_proj's q, k, v and r_proj's r_k = emb W_r^T in one
    launch; emb [M+L, d] (M+L rows of the position embedding), w_r [d, d].
    Returns (q, k, v, r_k)."""
    d = w_qkv.shape[1]
    dh = d // H
    if emb.dim() != 2 or emb.shape[1] != d:
        raise ValueError("emb must be [M+L, d]")
    Kr = emb.shape[0]
    _need(emb, "emb", (Kr, d), torch.bfloat16, h.device)
    _need(w_r, "w_r", (d, d), torch.bfloat16, h.device)
    if r_k is None:
        r_k = torch.empty((Kr, H, dh), dtype=torch.bfloat16, device=h.device)
    _need(r_k, "r_k", (Kr, H, dh), torch.bfloat16, h.device)
    q, k, v, (B, L, M) = _qkv_args(h, mem, w_qkv, H, q, k, v)
    if Kr != M + L:
        raise ValueError(f"emb has {Kr} rows, expected M+L = {M + L}")
    h_layout = 0 if h.dim() == 3 else 1
    mem_layout = 0 if mem.dim() == 3 else 1
    rc = _invoke(h.device, "txl_qkvr_proj", h.data_ptr(), h_layout, mem.data_ptr() if M > 0 else 0,
                 mem_layout, int(mem_start), w_qkv.data_ptr(), emb.data_ptr(), w_r.data_ptr(), B, L, M, H,
                 dh, q.data_ptr(), k.data_ptr(), v.data_ptr(), r_k.data_ptr(), _stream(stream, h.device))
    if rc != 0:
        raise TxlError(rc, "txl_qkvr_proj")
    return q, k, v, r_k


def linear(x, w, bias=None, resid=None, relu=False, out=None, stream=None):
    """txl_linear: out [B, T, N] = relu?(x W^T + bias) + resid; x [B, T, K]
    (rows) or [B, H, T, 64] (heads: read as [B, T, H*64]); w [N, K]; bias [N];
    resid [B, T, N] (may be ``out``).  bf16 CUDA tensors."""
    if x.dim() == 3:
        B, T, K = x.shape
        layout = 0
    elif x.dim() == 4:
        B, Hh, T, dh = x.shape
        if dh != 64:
            raise ValueError("the heads layout needs d_h = 64")
        K, layout = Hh * dh, 1
    else:
        raise ValueError("x must be [B, T, K] or [B, H, T, 64]")
    N = w.shape[0]
    _need(x, "x", tuple(x.shape), torch.bfloat16)
    _need(w, "w", (N, K), torch.bfloat16, x.device)
    if bias is not None:
        _need(bias, "bias", (N,), torch.bfloat16, x.device)
    if resid is not None:
        _need(resid, "resid", (B, T, N), torch.bfloat16, x.device)
    if out is None:
        out = torch.empty((B, T, N), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", (B, T, N), torch.bfloat16, x.device)
    rc = _invoke(x.device, "txl_linear", x.data_ptr(), layout, B, T, K, w.data_ptr(), N,
                           bias.data_ptr() if bias is not None else 0,
                           resid.data_ptr() if resid is not None else 0, int(bool(relu)),
                           out.data_ptr(), _stream(stream, x.device))
    if rc != 0:
        raise TxlError(rc, "txl_linear")
    return out


def layer_norm(x, gamma, beta, y=None, eps=1e-5, out=None, stream=None):
    """txl_layer_norm: LayerNorm(x + y) * gamma + beta over the last axis (y
    optional); bf16 CUDA tensors; out may be x or y."""
    d = x.shape[-1]
    rows = x.numel() // d
    _need(x, "x", tuple(x.shape), torch.bfloat16)
    if y is not None:
        _need(y, "y", tuple(x.shape), torch.bfloat16, x.device)
    _need(gamma, "gamma", (d,), torch.bfloat16, x.device)
    _need(beta, "beta", (d,), torch.bfloat16, x.device)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", tuple(x.shape), torch.bfloat16, x.device)
    rc = _invoke(x.device, "txl_layer_norm", x.data_ptr(), y.data_ptr() if y is not None else 0, gamma.data_ptr(),
                               beta.data_ptr(), rows, d, float(eps), out.data_ptr(),
                               _stream(stream, x.device))
    if rc != 0:
        raise TxlError(rc, "txl_layer_norm")
    return out


def r_proj(emb, w_r, H, out=None, stream=None):
    """txl_r_proj: r_k [K, H, d_h] = emb [K, d] W_r^T; bf16 CUDA tensors."""
    K, d = emb.shape
    dh = d // H
    _need(emb, "emb", (K, d), torch.bfloat16)
    _need(w_r, "w_r", (d, d), torch.bfloat16, emb.device)
    if out is None:
        out = torch.empty((K, H, dh), dtype=torch.bfloat16, device=emb.device)
    _need(out, "r_k", (K, H, dh), torch.bfloat16, emb.device)
    rc = _invoke(emb.device, "txl_r_proj", emb.data_ptr(), w_r.data_ptr(), K, H, dh, out.data_ptr(), _stream(stream, emb.device))
    if rc != 0:
        raise TxlError(rc, "txl_r_proj")
    return out


def mem_update(mems: torch.Tensor, hids: torch.Tensor, stream=None, ext_len: int = 0) -> torch.Tensor:
    """Tail_M roll in place (txl_mem_update, or txl_mem_update_ext when
    ext_len > 0): mems [B,M,d] <- newest M rows of [mems; hids[:, :L-ext_len]],
    hids [B,L,d].  Returns mems."""
    if mems.dim() != 3 or hids.dim() != 3:
        raise ValueError("mems must be [B, M, d] and hids [B, L, d]")
    B, M, d = mems.shape
    L = hids.shape[1]
    _need(mems, "mems", (B, M, d), mems.dtype)
    _need(hids, "hids", (B, L, d), mems.dtype, mems.device)
    if ext_len:
        rc = _invoke(mems.device, "txl_mem_update_ext", mems.data_ptr(), hids.data_ptr(), B, L, M, d, int(ext_len),
                                       _dtype_code(mems), _stream(stream, mems.device))
        if rc != 0:
            raise TxlError(rc, "txl_mem_update_ext")
        return mems
    rc = _invoke(mems.device, "txl_mem_update", mems.data_ptr(), hids.data_ptr(), B, L, M, d, _dtype_code(mems),
                               _stream(stream, mems.device))
    if rc != 0:
        raise TxlError(rc, "txl_mem_update")
    return mems


def mem_ring_push(ring: torch.Tensor, hids: torch.Tensor, start: int, stream=None) -> int:
    """txl_mem_ring_push: ring [B, M, d] (logical row t at row (start+t) % M)
    takes the rows of hids [B, L, d]; returns the new start."""
    if ring.dim() != 3 or hids.dim() != 3:
        raise ValueError("ring must be [B, M, d] and hids [B, L, d]")
    B, M, d = ring.shape
    L = hids.shape[1]
    _need(ring, "ring", (B, M, d), ring.dtype)
    _need(hids, "hids", (B, L, d), ring.dtype, ring.device)
    new = ctypes.c_int(0)
    rc = _invoke(ring.device, "txl_mem_ring_push", ring.data_ptr(), hids.data_ptr(), B, L, M, d, int(start), ctypes.byref(new),
                                  _dtype_code(ring), _stream(stream, ring.device))
    if rc != 0:
        raise TxlError(rc, "txl_mem_ring_push")
    return int(new.value)


def mem_reset(mems: torch.Tensor, flags: torch.Tensor, stream=None) -> torch.Tensor:
    """txl_mem_reset: zeroes batch row b of mems (any contiguous [B, ...]
    layout) wherever flags[b] is set; flags is a bool or uint8 CUDA tensor
    [B].  Returns mems."""
    if mems.dim() < 2 or not mems.is_cuda or not mems.is_contiguous():
        raise ValueError("mems must be a contiguous CUDA tensor [B, ...]")
    B = mems.shape[0]
    d = mems.shape[-1]
    rows = mems.numel() // (B * d) if B * d else 0
    if flags.shape != (B,) or flags.device != mems.device or flags.dtype not in (torch.bool, torch.uint8):
        raise ValueError("flags must be a bool/uint8 tensor [B] on the memory's device")
    f = flags.contiguous()
    rc = _invoke(mems.device, "txl_mem_reset", mems.data_ptr(), f.data_ptr(), B, rows, d, _dtype_code(mems),
                              _stream(stream, mems.device))
    if rc != 0:
        raise TxlError(rc, "txl_mem_reset")
    return mems


def sync_status(stream=None, device=None) -> int:
    """Waits for the stream and returns (and clears) the device status code."""
    dev = device if device is not None else torch.cuda.current_device()
    return int(_invoke(dev, "txl_sync_status", _stream(stream, dev)))


def check_status(stream=None) -> None:
    rc = sync_status(stream)
    if rc != 0:
        raise TxlError(rc, "device status")


def bounds_status() -> tuple[int, int]:
    """txl_bounds_status: (status, first record) of a bounds-checked build;
    status TXL_ERR_UNSUPPORTED (-2) from the plain build."""
    w = ctypes.c_ulonglong(0)
    rc = load().txl_bounds_status(ctypes.byref(w))
    return int(rc), int(w.value)


def debug_inject(kind: int) -> None:
    rc = load().txl_debug_inject(int(kind))
    if rc != 0:
        raise TxlError(rc, "txl_debug_inject")
