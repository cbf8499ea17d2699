"""Plain fp64 CPU oracle for Transformer-XL relative attention and Tail_M.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library and never imports it.

Functions
---------
attn(q, k, v, r_k, u, vb, scale, ...)
    The relative attention forward, computed by ``txl_oracle.c`` with one
    loop per (query, key) pair and the four-term score a+b+c+d ("Transformer-XL"
    notes, zty624, section "Relative Positional Encoding"), the rectangular
    mask allow(i, j) <=> j <= M+i (same notes, section "Causal Mask With
    Memory") and the distance convention of the position sequence M+L-1..0
    ("Transformer-XL模型 核心源码阅读笔记", section "Build the model",
    MemTransformerLM._forward).
mem_update(mem, hid, mem_len, ext_len=0)
    Tail_M: keep the newest ``mem_len`` rows of [mem; hid] along the sequence
    axis, with the index arithmetic of MemTransformerLM._update_mems in the
    source-reading notes (end = mlen + max(0, qlen - ext_len),
    beg = max(0, end - mem_len)) and the batch-major layout of the
    "Transformer-XL" notes, section "Batched Tensor Contract".
qkv_proj(h, mem, w_qkv, n_head), r_proj(emb, w_r, n_head)
    The projections that feed the attention, as the source-reading notes
    write them (RelPartialLearnableMultiHeadAttn.forward: qkv_net applied to
    the concatenation cat = [mems; w] along the sequence axis, its output
    chunked into q, k, v and viewed as heads; r_net applied to the position
    embedding): here literally a concatenation, an fp64 matrix product with
    the nn.Linear convention (output = input W^T) and a reshape into heads,
    batch-major as in the "Transformer-XL" notes' "Batched Tensor Contract".
sinusoid(pos, demb)
    Is NOT here: the sinusoid is input preparation and lives in the seeded
    workload module.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "txl_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into oracle/liboracle.so (portable flags:
    no -march, no FMA contraction, so x86 and Arm give the same results)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lib.oracle_attn_f64.argtypes = [dp, dp, dp, dp, dp, dp,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                            dp, dp, ip, ctypes.c_int, ctypes.c_int]
            lib.oracle_attn_f64.restype = ctypes.c_int
            lib.oracle_attn_f64_ex.argtypes = [dp, dp, dp, dp, dp, dp,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                               ctypes.c_int, ctypes.c_int,
                                               dp, dp, ip, ctypes.c_int, ctypes.c_int]
            lib.oracle_attn_f64_ex.restype = ctypes.c_int
            lib.oracle_num_cores.argtypes = []
            lib.oracle_num_cores.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact conversion to a contiguous fp64 numpy array (bf16/fp32 -> fp64 is exact)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_cores() -> int:
    return int(_load().oracle_num_cores())


def attn(q, k, v, r_k, u, vb, scale: float, pairs=None, want_scores: bool = False,
         nthreads: int = 0, same_length: bool = False, mem_len: int | None = None):
    """Relative attention forward in fp64.

    q [B,H,L,dh]; k, v [B,H,M+L,dh]; r_k [M+L,H,dh] (row r <-> distance
    M+L-1-r); u, vb [H,dh].  ``pairs`` optionally lists flat b*H+h indices to
    compute (other rows of the result are NaN).  Returns ``out`` [B,H,L,dh]
    or ``(out, scores)`` with scores [B,H,L,M+L] (-inf where masked).
    ``same_length`` adds the source notes' lower mask (every query sees the
    same number of keys) for the configured ``mem_len`` (default: M).
    """
    q, k, v, r_k, u, vb = (_f64(t) for t in (q, k, v, r_k, u, vb))
    B, H, L, dh = q.shape
    K = k.shape[2]
    M = K - L
    if k.shape != (B, H, K, dh) or v.shape != k.shape:
        raise ValueError("k, v must be [B,H,M+L,dh]")
    if r_k.shape != (K, H, dh) or u.shape != (H, dh) or vb.shape != (H, dh):
        raise ValueError("r_k must be [M+L,H,dh]; u, vb [H,dh]")
    out = np.full((B, H, L, dh), np.nan)
    scores = np.full((B, H, L, K), np.nan) if want_scores else None
    if pairs is not None:
        parr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32))
        if parr.size and (parr.min() < 0 or parr.max() >= B * H):
            raise ValueError("pair index out of range")
        pp = parr.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
        npairs = int(parr.size)
    else:
        parr, pp, npairs = None, None, 0
    rc = _load().oracle_attn_f64_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r_k), _ptr(u), _ptr(vb),
        B, H, L, M, dh, float(scale), int(bool(same_length)), int(M if mem_len is None else mem_len),
        _ptr(out),
        _ptr(scores) if scores is not None else None,
        pp, npairs, int(nthreads))
    if rc < 0:
        raise RuntimeError(f"oracle_attn_f64 failed ({rc})")
    return (out, scores) if want_scores else out


def mem_update(mem, hid, mem_len: int, ext_len: int = 0) -> np.ndarray:
    """Tail_M of [mem; hid] along axis 1 (batch-major [B, len, d]).

    Works on any dtype bit-for-bit: it only slices.  ``mem`` may hold fewer
    than ``mem_len`` rows (the growth phase); the result holds
    min(mem_len, mlen + qlen - ext_len) rows.
    """
    mem = np.asarray(mem)
    hid = np.asarray(hid)
    mlen, qlen = mem.shape[1], hid.shape[1]
    if mem_len == 0:
        return hid[:, :0].copy()
    end = mlen + max(0, qlen - ext_len)
    beg = max(0, end - mem_len)
    cat = np.concatenate([mem, hid], axis=1)
    return np.ascontiguousarray(cat[:, beg:end])


def mem_reset(mem, flags) -> np.ndarray:
    """Per-row memory reset ("Transformer-XL" notes, section "Batched
    Streams": rows whose stream enters a new document get zeros; the flag is
    per batch row).  mem [B, ...] of any dtype, flags [B]; bit-exact."""
    out = np.array(mem, copy=True)
    out[np.asarray(flags).astype(bool)] = 0
    return out


def _heads(x: np.ndarray, n_head: int) -> np.ndarray:
    """[B, T, n_head*d_head] -> [B, n_head, T, d_head]."""
    B, T, d = x.shape
    return x.reshape(B, T, n_head, d // n_head).transpose(0, 2, 1, 3).copy()


def qkv_proj(h, mem, w_qkv, n_head: int):
    """q from the current segment only, k and v from [mem; h]; w_qkv [3d, d]
    stacks W_q, W_k, W_v (output = input W^T).  Returns fp64 q [B,H,L,dh],
    k, v [B,H,M+L,dh]."""
    h64, m64, w64 = _f64(h), _f64(mem), _f64(w_qkv)
    d = h64.shape[2]
    cat = np.concatenate([m64, h64], axis=1)
    wq, wk, wv = w64[:d], w64[d:2 * d], w64[2 * d:]
    q = _heads(h64 @ wq.T, n_head)
    k = _heads(cat @ wk.T, n_head)
    v = _heads(cat @ wv.T, n_head)
    return q, k, v


def r_proj(emb, w_r, n_head: int):
    """r_k [K, H, dh] = emb [K, d] W_r^T (fp64)."""
    e64, w64 = _f64(emb), _f64(w_r)
    K, d = e64.shape
    return (e64 @ w64.T).reshape(K, n_head, d // n_head)


# ---------------------------------------------------------------------------
# The rest of a decoder layer ("Transformer-XL模型 核心源码阅读笔记":
# RelPartialLearnableMultiHeadAttn.forward after the attention, PositionwiseFF,
# RelPartialLearnableDecoderLayer).  Row-major [B, T, d] activations, fp64.
# ---------------------------------------------------------------------------
def layer_norm(x, gamma, beta, eps: float = 1e-5) -> np.ndarray:
    """nn.LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * gamma +
    beta with the biased (population) variance of each row."""
    x64 = _f64(x)
    mean = x64.mean(axis=-1, keepdims=True)
    var = ((x64 - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x64 - mean) / np.sqrt(var + eps) * _f64(gamma) + _f64(beta)


def linear(x, w, b=None) -> np.ndarray:
    """nn.Linear: x W^T (+ b); w [N, K]."""
    y = _f64(x) @ _f64(w).T
    return y if b is None else y + _f64(b)


def merge_heads(o) -> np.ndarray:
    """[B, H, T, d_h] -> [B, T, H*d_h] (attn_vec of the notes)."""
    o64 = _f64(o)
    B, H, T, dh = o64.shape
    return o64.transpose(0, 2, 1, 3).reshape(B, T, H * dh)


def attn_block_out(w, attn_vec, w_o, ln_g, ln_b, pre_lnorm: bool) -> np.ndarray:
    """After the attention: attn_out = o_net(attn_vec) (no bias); post-norm
    LN(w + attn_out), pre-norm w + attn_out."""
    attn_out = linear(attn_vec, w_o)
    return _f64(w) + attn_out if pre_lnorm else layer_norm(_f64(w) + attn_out, ln_g, ln_b)


def pos_ff(x, w1, b1, w2, b2, ln_g, ln_b, pre_lnorm: bool) -> np.ndarray:
    """PositionwiseFF: CoreNet = Linear(d, d_inner) -> ReLU -> Linear(d_inner,
    d); post-norm LN(x + core(x)), pre-norm x + core(LN(x))."""
    x64 = _f64(x)
    inp = layer_norm(x64, ln_g, ln_b) if pre_lnorm else x64
    core = linear(np.maximum(linear(inp, w1, b1), 0.0), w2, b2)
    return x64 + core if pre_lnorm else layer_norm(x64 + core, ln_g, ln_b)



# ---------------------------------------------------------------------------
# Backward of the attention ("Transformer-XL" notes, zty624: training with a
# stop-gradient memory -- the memory enters the segment as a constant input,
# so gradients stop at the memory rows' keys and values and never reach the
# earlier segment).  Derived from the forward definition above:
#   s_ij  = scale ((q_i + u) . k_j + (q_i + v) . R_dist(i,j))   (allowed pairs)
#   P     = softmax_j(s),  O_i = sum_j P_ij V_j
#   dV_j  = sum_i P_ij dO_i
#   dP_ij = dO_i . V_j,    dS_ij = P_ij (dP_ij - dO_i . O_i)
#   dq_i  = scale sum_j dS_ij (k_j + R_dist)
#   dk_j  = scale sum_i dS_ij (q_i + u)
#   dR_r  = scale sum over pairs with R row r of dS_ij (q_i + v)
#   du    = scale sum_ij dS_ij k_j,   dv = scale sum_ij dS_ij R_dist
# (u, v and R are shared by the batch; u, v per head.)  fp64, one query row
# at a time.
# ---------------------------------------------------------------------------
def attn_bwd(q, k, v, r_k, u, vb, scale: float, dout, same_length: bool = False,
             mem_len: int | None = None):
    """Returns dict of fp64 gradients dq [B,H,L,dh], dk, dv [B,H,M+L,dh],
    dr [M+L,H,dh], du, dvb [H,dh] of sum(out * dout)."""
    q, k, v, r, u, vb, g = (_f64(t) for t in (q, k, v, r_k, u, vb, dout))
    B, H, L, dh = q.shape
    K = k.shape[2]
    M = K - L
    if same_length:
        ml = M if mem_len is None else mem_len
        mask_len = K - ml
        shift = L - mask_len if mask_len > 0 else L
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dr = np.zeros_like(r)
    du = np.zeros_like(u)
    dvb = np.zeros_like(vb)
    j = np.arange(K)
    for b in range(B):
        for h in range(H):
            for i in range(L):
                allow = (j - i) <= M
                if same_length:
                    allow &= (j - i) > -shift
                js = j[allow]
                rows = K - 1 - (M + i - js)          # R row of each allowed pair
                Rj = r[rows, h]                        # [n, dh]
                kj = k[b, h, js]
                s = scale * ((kj @ (q[b, h, i] + u[h])) + (Rj @ (q[b, h, i] + vb[h])))
                p = np.exp(s - s.max())
                p /= p.sum()
                o = p @ v[b, h, js]
                dP = v[b, h, js] @ g[b, h, i]
                dS = p * (dP - g[b, h, i] @ o)
                dv[b, h, js] += np.outer(p, g[b, h, i])
                dq[b, h, i] = scale * (dS @ (kj + Rj))
                dk[b, h, js] += scale * np.outer(dS, q[b, h, i] + u[h])
                np.add.at(dr[:, h], rows, scale * np.outer(dS, q[b, h, i] + vb[h]))
                du[h] += scale * (dS @ kj)
                dvb[h] += scale * (dS @ Rj)
    return {"dq": dq, "dk": dk, "dv": dv, "dr": dr, "du": du, "dvb": dvb}
