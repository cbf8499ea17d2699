"""GB300-native (sm_103a) Transformer-XL relative attention over a per-layer
recurrence memory.

Public API (all computation runs in libtxl.so's CUDA kernels):
    attn_fwd, attn_fwd_ws, attn_workspace_bytes   relative attention forward
    attn_fwd_lse                                  the same, also returning the rows' log2-sum-exp
    attn_fwd_noalloc                              the same with the library's static scratch
    attn_bwd, attn_bwd_workspace_bytes            its gradients (stop-gradient memory; tensor cores)
    mem_update, mem_reset                         Tail_M memory roll (ext_len), per-row reset, in place
    mem_ring_push                                 ring-buffer memory update (qkv_proj reads the ring)
    qkv_proj, r_proj                              head-split input projections (tensor cores)
    qkvr_proj                                     both in one launch
    linear, layer_norm                            o_net / feed-forward GEMMs, fused residual LayerNorm
    sync_status, check_status                     device status word
    bounds_status                                 first out-of-range access (bounds-checked build)
    SegmentDriver                                 multi-segment, multi-layer driver (caller's projections)
    AttnStack                                     the same with the library's projections
    DecoderStack                                  full decoder layers (attention, o_net, LayerNorm, feed-forward)
"""
from ._lib import (TXL_BF16, TXL_F32, TxlError, attn_bwd, attn_bwd_workspace_bytes, attn_fwd, attn_fwd_lse, attn_fwd_noalloc, attn_fwd_ws,
                   attn_workspace_bytes, bounds_status,
                   check_status, debug_inject, header_functions, layer_norm, linear, load, mem_reset, mem_ring_push, mem_update, qkv_proj, qkvr_proj, r_proj,
                   status_string,
                   sync_status, version, LIB_PATH)
from .driver import AttnStack, DecoderStack, SegmentDriver

__all__ = ["TXL_BF16", "TXL_F32", "TxlError", "attn_bwd", "attn_bwd_workspace_bytes", "attn_fwd", "attn_fwd_lse", "attn_fwd_noalloc", "attn_fwd_ws",
           "attn_workspace_bytes", "bounds_status",
           "check_status", "debug_inject", "header_functions", "layer_norm", "linear", "load", "mem_reset", "mem_ring_push", "mem_update", "qkv_proj", "qkvr_proj", "r_proj",
           "status_string", "sync_status", "version", "SegmentDriver", "AttnStack", "DecoderStack", "LIB_PATH"]
