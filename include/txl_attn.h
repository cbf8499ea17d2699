/*
 * txl_attn.h -- C ABI of the GB300 (sm_103a) Transformer-XL relative
 * attention library (libtxl.so).
 *
 * The operation is relative multi-head attention over a per-layer recurrence
 * memory, as defined by:
 *   - "Transformer-XL" course notes (zty624.github.io), sections
 *     "Segment-Level Recurrence", "Batched Tensor Contract",
 *     "Causal Mask With Memory", "Relative Positional Encoding" and
 *     "Relative Shift Trick";
 *   - "Transformer-XL模型 核心源码阅读笔记" (CSDN source-reading notes),
 *     section "Build the model": RelPartialLearnableMultiHeadAttn.forward and
 *     MemTransformerLM._forward / _update_mems.
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, contiguous, row-major, on the current CUDA
 *     device; every pointer argument is a DEVICE pointer.  The caller owns
 *     every buffer; the library never allocates, frees or retains them.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise the host, except
 *     txl_sync_status().
 *   - Return value: TXL_OK (0) on success, a negative txl_status otherwise.
 *     Argument errors are detected on the host before anything is launched.
 *     No kernel traps or asserts: a device-side wait that runs past its
 *     time limit records TXL_ERR_DEVICE_TIMEOUT in a device status word,
 *     which txl_sync_status() reports and clears.
 *   - dtype: TXL_BF16 (inputs and output bf16, fp32 accumulation on the
 *     tensor cores) or TXL_F32 (inputs and output fp32, fp32 CUDA-core path).
 */
#ifndef TXL_ATTN_H
#define TXL_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum txl_dtype {
    TXL_F32 = 0,
    TXL_BF16 = 1
};

enum txl_status {
    TXL_OK = 0,
    TXL_ERR_INVALID_ARG = -1,    /* null pointer, B/H/L <= 0, M < 0, bad dtype */
    TXL_ERR_UNSUPPORTED = -2,    /* a size the library has no kernel for (see each call) */
    TXL_ERR_MISALIGNED = -3,     /* a base pointer is not 16-byte aligned */
    TXL_ERR_ALIAS = -4,          /* an output overlaps an input it must not overlap */
    TXL_ERR_LAUNCH = -5,         /* the CUDA launch itself failed */
    TXL_ERR_DEVICE_TIMEOUT = -6, /* a bounded device-side wait expired (reported by txl_sync_status) */
    TXL_ERR_WORKSPACE = -7,      /* workspace pointer null/misaligned or smaller than required */
    TXL_ERR_CUDA = -8,           /* a CUDA runtime/driver call failed (e.g. tensor-map encoding) */
    TXL_ERR_SCRATCH_LIMIT = -9,  /* the call needs more scratch than txl_attn_fwd_noalloc holds */
    TXL_ERR_OUT_OF_BOUNDS = -10  /* a bounds-checked build skipped an out-of-range access */
};

/*
 * Relative attention forward for one layer and one segment.
 *
 *   q      [B, H, L, d_h]      queries of the current segment only
 *   k, v   [B, H, M+L, d_h]    keys / values: rows 0..M-1 are the memory
 *                              (previous segment, stop-gradient), rows
 *                              M..M+L-1 the current segment
 *   r_k    [M+L, H, d_h]       projected sinusoid position table; row r holds
 *                              relative distance M+L-1-r (distance 0 last)
 *   u_bias [H, d_h]            global content bias u   (r_w_bias)
 *   v_bias [H, d_h]            global position bias v  (r_r_bias)
 *   out    [B, H, L, d_h]      result
 *
 * For query i in [0,L) and key j in [0,M+L):
 *   visible(i,j) <=> j <= M+i          (all memory keys, causal current keys)
 *   s(i,j) = scale * ((q_i+u).k_j + (q_i+v).r_k[M+L-1-(M+i-j)])
 *   out_i  = sum_j softmax_j(s(i,.)) v_j   over visible j only.
 * M = 0 is ordinary causal attention with a relative bias.
 *
 * bf16: d_h must be 64 (TXL_ERR_UNSUPPORTED otherwise); fp32: 1 <= d_h <= 256.
 * All pointers 16-byte aligned (TXL_ERR_MISALIGNED).  `out` must not overlap
 * any input (TXL_ERR_ALIAS).  This entry point allocates nothing and never
 * splits the keys of a query tile across CTAs; txl_attn_fwd_ws may.
 */
int txl_attn_fwd(const void* q, const void* k, const void* v, const void* r_k,
                 const void* u_bias, const void* v_bias,
                 int B, int H, int L, int M, int d_h, float scale, void* out,
                 int dtype, void* stream);

/*
 * txl_attn_fwd_ex: txl_attn_fwd with the same_length mask of
 * "Transformer-XL模型 核心源码阅读笔记" (MemTransformerLM._forward): every query
 * attends over the same number of keys.  With klen = M+L and mask_len = klen -
 * mem_len, query i additionally ignores keys j <= i - mask_shift_len, where
 * mask_shift_len = L - mask_len if mask_len > 0, else L; when M = mem_len each
 * query sees its mem_len most recent positions, itself included.  mem_len is
 * the configured memory length (M <= mem_len; M < mem_len while the memory is
 * still filling), else TXL_ERR_INVALID_ARG.  Key tiles that no query of a
 * 128-row query tile sees are skipped.  same_length = 0 is txl_attn_fwd.
 * Everything else (layouts, sizes, errors) as for txl_attn_fwd.
 */
int txl_attn_fwd_ex(const void* q, const void* k, const void* v, const void* r_k,
                    const void* u_bias, const void* v_bias, int B, int H, int L, int M, int d_h,
                    float scale, int same_length, int mem_len, void* out, int dtype, void* stream);

/*
 * Scratch bytes txl_attn_fwd_ws needs for these sizes (0 when the call runs
 * without splitting the keys).  Never negative; 0 also for invalid sizes.
 */
size_t txl_attn_workspace_bytes(int B, int H, int L, int M, int d_h, int dtype);

/*
 * txl_attn_fwd with caller-provided scratch: `workspace` (device, 256-byte
 * aligned, at least txl_attn_workspace_bytes(...) bytes) holds the partial
 * results of the split-key path, which the bf16 kernel takes when the call has
 * fewer (b, h, 128-row query tile) items than the GPU has SMs: each item's key
 * tiles are split over several CTAs, each writes its unnormalised partial O
 * and (max, sum) per row, and a combine pass merges them (the online-softmax
 * merge).  Nothing in the workspace needs to start at zero; every value read
 * is written earlier in the same call.  With a size of 0 the workspace is not
 * touched and may be null.  The library allocates nothing.
 * TXL_ERR_WORKSPACE if the buffer is missing, misaligned or too small;
 * TXL_ERR_ALIAS if it overlaps q, k, v or out.  Concurrent calls must use
 * distinct workspaces.
 */
int txl_attn_fwd_ws(const void* q, const void* k, const void* v, const void* r_k,
                    const void* u_bias, const void* v_bias,
                    int B, int H, int L, int M, int d_h, float scale, void* out,
                    int dtype, void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of the static device scratch that txl_attn_fwd_noalloc uses.
 */
#define TXL_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * txl_attn_fwd_ws without a caller workspace and without any allocation: the
 * split-key path (see txl_attn_fwd_ws) takes its partial results from one
 * file-scope static device buffer of TXL_NOALLOC_SCRATCH_BYTES (16 MiB) per
 * device.  The library looks its device address up (cudaGetSymbolAddress)
 * on every call that is not inside a stream capture and keeps the last
 * address per device for calls made during a capture.  The pages have no
 * counterpart of this entry point: it exists for callers that cannot hand
 * out a workspace (for example a fixed launch sequence).
 *
 *   - Same arguments, results and errors as txl_attn_fwd_ws; a call whose
 *     txl_attn_workspace_bytes(...) exceeds TXL_NOALLOC_SCRATCH_BYTES returns
 *     TXL_ERR_SCRATCH_LIMIT and launches nothing.
 *   - Nothing in the scratch needs to start at zero: every value read is
 *     written earlier in the same call.
 *   - The first call on each device that needs scratch must not be inside a
 *     stream capture (there is no cached address yet: TXL_ERR_CUDA).  After
 *     cudaDeviceReset (or any teardown of the device's context) the module is
 *     loaded again at a new address: make one call outside a capture before
 *     capturing again, or a capture would launch on the stale address.
 *   - Calls that overlap in time on one device (different streams, or
 *     threads) share the buffer and race: order them, e.g. on one stream.
 *   - Calls that need no scratch (txl_attn_workspace_bytes(...) == 0) do not
 *     touch it.
 */
int txl_attn_fwd_noalloc(const void* q, const void* k, const void* v, const void* r_k,
                         const void* u_bias, const void* v_bias,
                         int B, int H, int L, int M, int d_h, float scale, void* out,
                         int dtype, void* stream);

/*
 * Projections feeding txl_attn_fwd, bf16 in and out, fp32 accumulation, on
 * the tensor cores ("Transformer-XL模型 核心源码阅读笔记",
 * RelPartialLearnableMultiHeadAttn.forward: qkv_net over the concatenation of
 * memory and current hidden states, r_net over the position embedding).
 *
 * txl_qkv_proj:
 *   h     [B, L, d]     current hidden states (layer input), d = H * d_h
 *   mem   [B, M, d]     the layer's memory (may be null when M = 0)
 *   w_qkv [3d, d]       stacked weights, rows [0,d) W_q, [d,2d) W_k, [2d,3d) W_v
 *                       (output = input x W^T, the nn.Linear layout)
 *   q     [B, H, L, d_h]      q = h W_q^T, split into heads
 *   k, v  [B, H, M+L, d_h]    rows 0..M-1 from mem, rows M.. from h, split into
 *                             heads (no [mem; h] concatenation is formed)
 * txl_r_proj:
 *   emb   [K, d]   position embedding rows (the sinusoid of distances K-1..0)
 *   w_r   [d, d]   W_r (nn.Linear layout)
 *   r_k   [K, H, d_h] = emb W_r^T (row-major [K, d])
 *
 * Supported sizes (TXL_ERR_UNSUPPORTED otherwise): d_h = 64, H a multiple of
 * 4, L, M and K multiples of 128 (M may be 0).  Pointers 16-byte aligned
 * (TXL_ERR_MISALIGNED); outputs must not overlap inputs (TXL_ERR_ALIAS).
 * Asynchronous on `stream`; nothing is allocated.  Bounded device waits
 * report TXL_ERR_DEVICE_TIMEOUT through txl_sync_status.
 */
int txl_qkv_proj(const void* h, const void* mem, const void* w_qkv, int B, int L, int M, int H,
                 int d_h, void* q, void* k, void* v, void* stream);

/*
 * txl_qkvr_proj: one layer's projections in one launch -- txl_qkv_proj_ring's
 * q, k, v (same arguments and contract) and txl_r_proj's r_k = emb W_r^T over
 * K = M + L rows of the position embedding emb [M+L, d] (same contract) --
 * dealt from one tile list, so the small position projection rides in the
 * q/k/v launch instead of occupying a few SMs of a launch of its own
 * ("Transformer-XL模型 核心源码阅读笔记", RelPartialLearnableMultiHeadAttn.forward:
 * w_heads = qkv_net(cat), r_head_k = r_net(r)).  r_k must not overlap any
 * other argument (TXL_ERR_ALIAS).
 */
int txl_qkvr_proj(const void* h, int h_layout, const void* mem, int mem_layout, int mem_start,
                  const void* w_qkv, const void* emb, const void* w_r, int B, int L, int M, int H,
                  int d_h, void* q, void* k, void* v, void* r_k, void* stream);

/*
 * txl_qkv_proj_ex: txl_qkv_proj with the layout of h and mem chosen per
 * argument.  TXL_LAYOUT_ROWS: [B, T, d] as above.  TXL_LAYOUT_HEADS:
 * [B, H, T, d_h], the layout txl_attn_fwd writes its output in, so a stack of
 * layers feeds one layer's attention output (and the memory rolled from it)
 * straight into the next layer's projections; row t of head h is columns
 * h*d_h .. h*d_h+d_h-1 of the row-major view.  Other layouts return
 * TXL_ERR_INVALID_ARG; sizes, alignment and aliasing as for txl_qkv_proj.
 */
#define TXL_LAYOUT_ROWS 0
#define TXL_LAYOUT_HEADS 1
int txl_qkv_proj_ex(const void* h, int h_layout, const void* mem, int mem_layout,
                    const void* w_qkv, int B, int L, int M, int H, int d_h, void* q, void* k,
                    void* v, void* stream);

/*
 * Ring-buffer memory (an alternative to the Tail_M copy): a memory
 * of M rows whose logical row t is stored at row (start + t) mod M.
 *
 * txl_qkv_proj_ring: txl_qkv_proj_ex reading mem as a ring starting at
 *   mem_start (0 <= mem_start < M, a multiple of 128: every 128-row tile of
 *   the ring is then contiguous; TXL_ERR_UNSUPPORTED otherwise).  Same result
 *   as txl_qkv_proj_ex on the logical (unrotated) memory.
 * txl_mem_ring_push: the ring counterpart of txl_mem_update.  For L < M the
 *   L rows of hids [B, L, d] overwrite the ring's L oldest rows (hids row r
 *   at ring row (start + r) mod M) and *new_start = (start + L) mod M: L rows
 *   are written instead of M moved.  For L >= M the ring is refilled with the
 *   newest M rows and *new_start = 0.  The logical memory afterwards equals
 *   txl_mem_update's result.  Arguments and errors as txl_mem_update, plus
 *   start in [0, M) (TXL_ERR_INVALID_ARG) and new_start a host pointer.
 */
int txl_qkv_proj_ring(const void* h, int h_layout, const void* mem, int mem_layout, int mem_start,
                      const void* w_qkv, int B, int L, int M, int H, int d_h, void* q, void* k,
                      void* v, void* stream);
int txl_mem_ring_push(void* ring, const void* hids, int B, int L, int M, int d, int start,
                      int* new_start, int dtype, void* stream);
int txl_r_proj(const void* emb, const void* w_r, int K, int H, int d_h, void* r_k, void* stream);

/*
 * txl_attn_bwd: gradients of sum(out * dout) for the attention of
 * txl_attn_fwd / txl_attn_fwd_ex (same inputs, same mask options), for
 * training with a stop-gradient memory ("Transformer-XL" notes: the memory is
 * a constant input of the segment; its rows' dk, dv are returned and the
 * caller drops them).  Inputs in dtype (TXL_BF16 or TXL_F32), d_h <= 256;
 * gradients in fp32, device buffers the call overwrites:
 *   dq [B, H, L, d_h], dk, dv [B, H, M+L, d_h], dr [M+L, H, d_h] (summed
 *   over the batch), du, dvb [H, d_h] (summed over batch and query rows).
 * P is recomputed from q, k, r_k, u, v (no forward state is kept).  CUDA-core
 * arithmetic with fp32 atomics for the summed gradients: a correctness path
 * whose summation order is not fixed.  Errors as txl_attn_fwd; gradient
 * buffers must not overlap the inputs or each other (TXL_ERR_ALIAS).
 */
int txl_attn_bwd(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                 const void* v_bias, const void* dout, int B, int H, int L, int M, int d_h, float scale,
                 int same_length, int mem_len, float* dq, float* dk, float* dv, float* dr, float* du,
                 float* dvb, int dtype, void* stream);

/*
 * txl_attn_bwd_ws: the gradients of txl_attn_bwd (same arguments, layouts,
 * outputs and errors) on the tensor cores, for bf16 inputs with d_h = 64 and
 * the plain causal mask with memory (same_length = 0).  Any other call needs
 * no workspace and runs txl_attn_bwd.
 *
 * The pass follows the derivative of the attention of "Transformer-XL模型 核心
 * 源码阅读笔记", section "Build the model" (RelPartialLearnableMultiHeadAttn.
 * forward: AC + shifted BD, masked softmax, P V) with the memory a constant
 * input ("Transformer-XL" notes, section "Segment-Level Recurrence"), in four
 * launches on `stream`: the forward kernel of txl_attn_fwd_lse writes the
 * output and each query row's log2-sum-exp into the workspace; a small
 * kernel computes D = dout . out per row, writes (q+u) and (q+v) scaled by
 * scale * log2 e in bf16 and zeroes dr, du, dvb; a query-major pass recomputes P, dP and dS
 * per 128-row query tile and writes dq and accumulates dr, du, dvb; a
 * key-major pass recomputes them per 128-key tile and writes dk, dv (it may
 * start on the SMs the query-major pass leaves; the call's last launch
 * completes after both).  dr, du and dvb are accumulated with fp32 atomics
 * (summation order not fixed); dq, dk and dv are written once per element.  Contractions in bf16 with fp32
 * accumulation: P and dS are rounded to bf16 before their products.
 *
 * workspace: device memory owned by the caller, 256-byte aligned, at least
 * txl_attn_bwd_workspace_bytes(...) bytes (0 when the call runs
 * txl_attn_bwd); it must not overlap an input or a gradient (TXL_ERR_ALIAS).
 * TXL_ERR_WORKSPACE when it is null, misaligned or too small.
 */
size_t txl_attn_bwd_workspace_bytes(int B, int H, int L, int M, int d_h, int dtype, int same_length);

/*
 * txl_attn_fwd_lse: txl_attn_fwd (bf16, d_h = 64) that also writes each query
 * row's log2-sum-exp of its scores, lse [B, H, L] fp32 (log2 units: with s_ij
 * the score of "Transformer-XL模型 核心源码阅读笔记", RelPartialLearnableMultiHead
 * Attn.forward, P_ij = 2^(s_ij log2 e - lse_i)), the state a backward pass
 * needs besides `out`.  lse: device memory, 16-byte aligned, not overlapping
 * any other argument (TXL_ERR_ALIAS); TXL_ERR_UNSUPPORTED for TXL_F32.
 *
 * txl_attn_bwd_saved: the gradients of txl_attn_bwd_ws from the forward's
 * saved state instead of a recomputed forward: out [B, H, L, d_h] (bf16) and
 * lse as written by txl_attn_fwd_lse for the same inputs, D = dout . out per
 * row.  bf16, d_h = 64, no same_length (TXL_ERR_UNSUPPORTED otherwise); the
 * workspace of txl_attn_bwd_workspace_bytes(..., same_length = 0); the
 * gradients must overlap neither the inputs, out, lse nor the workspace.
 */
int txl_attn_fwd_lse(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                     const void* v_bias, int B, int H, int L, int M, int d_h, float scale, void* out, float* lse,
                     int dtype, void* stream);
int txl_attn_bwd_saved(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                       const void* v_bias, const void* out, const float* lse, const void* dout, int B, int H, int L,
                       int M, int d_h, float scale, float* dq, float* dk, float* dv, float* dr, float* du,
                       float* dvb, int dtype, void* workspace, size_t ws_bytes, void* stream);
int txl_attn_bwd_ws(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                    const void* v_bias, const void* dout, int B, int H, int L, int M, int d_h, float scale,
                    int same_length, int mem_len, float* dq, float* dk, float* dv, float* dr, float* du,
                    float* dvb, int dtype, void* workspace, size_t ws_bytes, void* stream);

/*
 * The rest of a decoder layer ("Transformer-XL模型 核心源码阅读笔记":
 * RelPartialLearnableMultiHeadAttn.forward after the attention, PositionwiseFF,
 * RelPartialLearnableDecoderLayer), bf16 with fp32 accumulation:
 *
 * txl_linear: out [B, T, N] = relu?(x W^T + bias) + resid (nn.Linear layout,
 *   w [N, K]); x [B, T, K] (TXL_LAYOUT_ROWS) or [B, K/64, T, 64]
 *   (TXL_LAYOUT_HEADS: an attention output read directly as attn_vec, the
 *   o_net input); bias [N] and resid [B, T, N] may be null.  Covers o_net
 *   (no bias), the two CoreNet layers (bias, ReLU on the first) and, in the
 *   pre-norm layer, their residual adds.  T a multiple of 128, K of 64, N of
 *   256 (TXL_ERR_UNSUPPORTED); out may be resid itself, no other overlap
 *   (TXL_ERR_ALIAS).
 * txl_layer_norm: out [rows, d] = LayerNorm(x + y) * gamma + beta over each
 *   row (y may be null; nn.LayerNorm: biased variance, eps inside the square
 *   root).  d in {256, 512, 768, 1024, 1536, 2048}; out may be x or y.
 *
 * All pointers are device pointers, 16-byte aligned (TXL_ERR_MISALIGNED).
 * Asynchronous on `stream`; nothing is allocated.
 */
int txl_linear(const void* x, int x_layout, int B, int T, int K, const void* w, int N,
               const void* bias, const void* resid, int relu, void* out, void* stream);
int txl_layer_norm(const void* x, const void* y, const void* gamma, const void* beta, long long rows,
                   int d, float eps, void* out, void* stream);

/*
 * Tail_M memory roll, in place ("Transformer-XL" notes, section
 * "Segment-Level Recurrence": M_{tau+1} = Tail_M([M_tau; H_tau]); source notes
 * MemTransformerLM._update_mems with ext_len = 0 and a full memory).
 *
 *   mems [B, M, d]   memory of one layer, overwritten with the newest M rows
 *                    of the sequence-axis concatenation [mems; hids]
 *   hids [B, L, d]   hidden states of the current segment (layer input)
 *
 * When L >= M the result is hids[:, L-M:]; when L < M it is
 * [mems[:, L:]; hids].  Bit-exact copy for any element type; dtype only
 * fixes the element size (TXL_BF16: 2 bytes, TXL_F32: 4 bytes).  M = 0 is a
 * no-op.  `mems` must not overlap `hids` (TXL_ERR_ALIAS).  Any alignment is
 * accepted; 16-byte aligned rows of a multiple of 16 bytes take the
 * vectorised path.
 */
int txl_mem_update(void* mems, const void* hids, int B, int L, int M, int d,
                   int dtype, void* stream);

/*
 * txl_mem_update_ext: txl_mem_update keeping the last ext_len rows of hids
 * out of the memory ("Transformer-XL模型 核心源码阅读笔记",
 * MemTransformerLM._update_mems: the cached span of [mems; hids] ends ext_len
 * rows before its end, those rows serving as extended context of the next
 * segment instead).  The result is the Tail_M roll with hids[:, :L-ext_len]
 * (an unchanged memory when ext_len >= L); hids is still [B, L, d].
 * ext_len < 0 returns TXL_ERR_INVALID_ARG.  ext_len = 0 is txl_mem_update.
 *
 * txl_mem_reset: mems [B, rows, d] (any layout whose batch rows are
 * contiguous, e.g. [B, H, M, d_h] with rows = H*M, d = d_h); every batch row
 * b with flags[b] != 0 (flags: B bytes in device memory) is set to zero bits
 * ("Transformer-XL" notes, section "Batched Streams": a row whose stream
 * enters a new document gets an empty memory; the flag is per row, not per
 * batch).  Other rows are untouched.  Asynchronous on `stream`.
 */
int txl_mem_update_ext(void* mems, const void* hids, int B, int L, int M, int d, int ext_len,
                       int dtype, void* stream);
int txl_mem_reset(void* mems, const void* flags, int B, int rows, int d, int dtype, void* stream);

/*
 * Waits for `stream`, then reports and clears the device status word:
 * TXL_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, TXL_ERR_CUDA if the stream reports a CUDA error, TXL_OK otherwise.
 */
int txl_sync_status(void* stream);

/*
 * Bounds-checked builds (the library compiled with -DTXL_CHECKED, shipped as
 * libtxl_checked.so beside libtxl.so): every kernel routes its computed
 * global-memory indexes and shared-memory addresses through a check; an
 * access outside its buffer is skipped, never performed, and the first such
 * access per source file is recorded (no trap, no fault).  TMA copies are
 * bounded by their tensor maps in hardware and are not re-checked.
 * txl_bounds_status synchronises the device, then returns TXL_OK when no
 * access was out of range since the last call, or TXL_ERR_OUT_OF_BOUNDS with
 * the first record in *first: bit 63 set, bits 40..62 the check site (the
 * hundreds digit names the source file), bits 0..39 the offending index
 * (mod 2^40).  The records are cleared.  TXL_ERR_UNSUPPORTED from a library
 * built without checks.  A debugging aid, not for production launches.
 */
int txl_bounds_status(unsigned long long* first);

/* Human-readable name of a txl_status value (static string). */
const char* txl_status_string(int status);

/* ABI version: (major << 16) | minor. */
int txl_version(void);

/*
 * Test hook for the failure-detection path.  kind = 1 makes the NEXT bf16
 * attention launch made by the calling host thread withhold one internal
 * completion signal, so its waiting warps hit their time limit, record
 * TXL_ERR_DEVICE_TIMEOUT and exit cleanly (the GPU context stays usable).
 * kind = 0 clears it.  The hook is per host thread (launches from other
 * threads never consume it) and disarms itself after one launch.  Not for
 * production use.
 */
int txl_debug_inject(int kind);

#ifdef __cplusplus
}
#endif

#endif /* TXL_ATTN_H */
