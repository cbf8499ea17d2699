// extern "C" entry points of libtxl.so (declared in include/txl_attn.h):
// argument validation on the host, then one asynchronous launch on the
// caller's stream.  Nothing here allocates device memory.
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "proj_gemm.h"
#include "txl_attn.h"
#include "txl_device.cuh"

namespace txl {
__device__ int g_dev_status = 0;

cudaError_t launch_tail_m(void* mem, const void* hid, int B, int L, int L_stride, int M,
                          size_t row_bytes, cudaStream_t stream);
cudaError_t launch_mem_reset(void* mem, const unsigned char* flags, int B, long long per_b_bytes,
                             cudaStream_t stream);
cudaError_t launch_ring_push(void* ring, const void* hid, int B, int L, int M, int start,
                             size_t row_bytes, cudaStream_t stream);
cudaError_t launch_attn_bwd_simt(const void* q, const void* k, const void* v, const void* r,
                                 const void* ub, const void* vb, const void* dout, int bf16, int B,
                                 int H, int L, int M, int dh, float scale, int lo_shift, float* dq,
                                 float* dk, float* dv, float* dr, float* du, float* dvb,
                                 cudaStream_t stream);
cudaError_t launch_layer_norm(const void* x, const void* y, const void* gamma, const void* beta,
                              long long rows, int d, float eps, void* out, cudaStream_t stream);
cudaError_t launch_attn_simt_f32(const float* q, const float* k, const float* v, const float* r,
                                 const float* ub, const float* vb, int B, int H, int L, int M,
                                 int dh, float scale, int lo_shift, float* out, cudaStream_t stream);
cudaError_t launch_attn_tc_bf16(const void* q, const void* k, const void* v, const void* r,
                                const void* ub, const void* vb, int B, int H, int L, int M,
                                float scale, int lo_shift, void* out, void* workspace, int inject,
                                int* status, cudaStream_t stream);
size_t attn_tc_bf16_workspace_bytes(int B, int H, int L, int M);
cudaError_t launch_attn_tc_bf16_lse(const void* q, const void* k, const void* v, const void* r, const void* ub,
                                    const void* vb, int B, int H, int L, int M, float scale, int lo_shift,
                                    void* out, float* lse, int* status, cudaStream_t stream);
cudaError_t launch_attn_bwd_tc(const void* q, const void* k, const void* v, const void* r, const void* ub,
                               const void* vb, const void* out, const float* lse, const void* dout, int B, int H,
                               int L, int M, float scale, float* dq, float* dk, float* dv, float* dr, float* du,
                               float* dvb, void* workspace, int* status, cudaStream_t stream);
size_t attn_bwd_tc_workspace_bytes(int B, int H, int L, int M);

// first bounds violation recorded by each translation unit (bounds-checked
// builds; 0 otherwise), read and cleared
unsigned long long bounds_word_attn_simt();
unsigned long long bounds_word_attn_tc();
unsigned long long bounds_word_attn_bwd();
unsigned long long bounds_word_attn_bwd_tc();
unsigned long long bounds_word_mem_update();
unsigned long long bounds_word_layer_norm();
unsigned long long bounds_word_proj_gemm();

}  // namespace txl

namespace {

// Scratch of txl_attn_fwd_noalloc: one static buffer per device (a module
// global exists once per device context).
__device__ __align__(256) unsigned char g_noalloc_scratch[TXL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Address of the static scratch on the current device.  Outside a stream
// capture it is looked up on every call (cheap), so a context torn down and
// rebuilt (cudaDeviceReset) never leaves a stale address in use; inside a
// capture, where the lookup may not run, the address cached by the last
// lookup on this device is used.
void* noalloc_scratch(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

// Test hook of txl_debug_inject: per host thread, consumed by the next
// bf16 attention launch of the same thread.
thread_local int g_inject = 0;

// Device address of the status word on the current device (looked up per
// call: cheap, and correct when the caller switches devices).
int* dev_status_ptr() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, txl::g_dev_status) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

int elem_size(int dtype) { return dtype == TXL_F32 ? 4 : (dtype == TXL_BF16 ? 2 : 0); }

int check_attn_args(const void* q, const void* k, const void* v, const void* r_k,
                    const void* u_bias, const void* v_bias, int B, int H, int L, int M, int d_h,
                    const void* out, int dtype) {
    const int es = elem_size(dtype);
    if (!es) return TXL_ERR_INVALID_ARG;
    if (!q || !k || !v || !r_k || !u_bias || !v_bias || !out) return TXL_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || L <= 0 || M < 0 || d_h <= 0) return TXL_ERR_INVALID_ARG;
    if (dtype == TXL_BF16 && d_h != 64) return TXL_ERR_UNSUPPORTED;
    if (dtype == TXL_F32 && d_h > 256) return TXL_ERR_UNSUPPORTED;
    // index arithmetic in the kernels uses 32-bit row counts per (b, h)
    const long long K = (long long)M + L;
    if (K >= (1ll << 30) || (long long)B * H >= (1ll << 30)) return TXL_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(r_k) || !aligned16(u_bias) ||
        !aligned16(v_bias) || !aligned16(out))
        return TXL_ERR_MISALIGNED;
    const size_t nq = (size_t)B * H * L * d_h * es;
    const size_t nkv = (size_t)B * H * K * d_h * es;
    const size_t nr = (size_t)K * H * d_h * es;
    const size_t nb = (size_t)H * d_h * es;
    if (overlap(out, nq, q, nq) || overlap(out, nq, k, nkv) || overlap(out, nq, v, nkv) ||
        overlap(out, nq, r_k, nr) || overlap(out, nq, u_bias, nb) || overlap(out, nq, v_bias, nb))
        return TXL_ERR_ALIAS;
    return TXL_OK;
}

// Arguments of both backward entry points (gradients fp32, inputs in dtype).
int check_bwd_args(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                   const void* v_bias, const void* dout, int B, int H, int L, int M, int d_h, int same_length,
                   int mem_len, const float* dq, const float* dk, const float* dv, const float* dr,
                   const float* du, const float* dvb, int dtype) {
    const int es = elem_size(dtype);
    if (!es) return TXL_ERR_INVALID_ARG;
    if (!q || !k || !v || !r_k || !u_bias || !v_bias || !dout || !dq || !dk || !dv || !dr || !du || !dvb)
        return TXL_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || L <= 0 || M < 0 || d_h <= 0) return TXL_ERR_INVALID_ARG;
    if (same_length && (mem_len < M || mem_len >= (1 << 30))) return TXL_ERR_INVALID_ARG;
    if (d_h > 256) return TXL_ERR_UNSUPPORTED;
    const long long K = (long long)M + L;
    if (K >= (1ll << 30) || (long long)B * H * K * d_h >= (1ll << 40)) return TXL_ERR_UNSUPPORTED;
    const void* ins[7] = {q, k, v, r_k, u_bias, v_bias, dout};
    const void* outs[6] = {dq, dk, dv, dr, du, dvb};
    for (const void* p : ins)
        if (!aligned16(p)) return TXL_ERR_MISALIGNED;
    for (const void* p : outs)
        if (!aligned16(p)) return TXL_ERR_MISALIGNED;
    const size_t nq = (size_t)B * H * L * d_h, nkv = (size_t)B * H * K * d_h, nr = (size_t)K * H * d_h,
                 nb = (size_t)H * d_h;
    const size_t in_n[7] = {nq * es, nkv * es, nkv * es, nr * es, nb * es, nb * es, nq * es};
    const size_t out_n[6] = {nq * 4, nkv * 4, nkv * 4, nr * 4, nb * 4, nb * 4};
    for (int o = 0; o < 6; ++o) {
        for (int i2 = 0; i2 < 7; ++i2)
            if (overlap(outs[o], out_n[o], ins[i2], in_n[i2])) return TXL_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 6; ++o2)
            if (overlap(outs[o], out_n[o], outs[o2], out_n[o2])) return TXL_ERR_ALIAS;
    }
    return TXL_OK;
}

// No lower key bound: the plain causal mask with memory.
constexpr int kNoLowerBound = 1 << 30;

// same_length (source-reading notes, MemTransformerLM._forward): with klen =
// M+L and mask_len = klen - mem_len, query i also ignores keys j <= i -
// mask_shift_len, where mask_shift_len = L - mask_len if mask_len > 0, else L.
int lower_shift(int same_length, int L, int M, int mem_len) {
    if (!same_length) return kNoLowerBound;
    const long long mask_len = (long long)M + L - mem_len;
    return mask_len > 0 ? (int)(L - mask_len) : L;
}

int launch_attn(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                const void* v_bias, int B, int H, int L, int M, int d_h, float scale, void* out,
                int dtype, void* workspace, void* stream, int lo_shift = kNoLowerBound) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == TXL_BF16) {
        int* status = dev_status_ptr();
        if (!status) return TXL_ERR_CUDA;
        const int inject = g_inject;
        g_inject = 0;
        e = txl::launch_attn_tc_bf16(q, k, v, r_k, u_bias, v_bias, B, H, L, M, scale, lo_shift, out,
                                     workspace, inject, status, st);
        if (e == cudaErrorInvalidValue) return TXL_ERR_CUDA;  // tensor-map encoding failed
    } else {
        e = txl::launch_attn_simt_f32(
            static_cast<const float*>(q), static_cast<const float*>(k),
            static_cast<const float*>(v), static_cast<const float*>(r_k),
            static_cast<const float*>(u_bias), static_cast<const float*>(v_bias), B, H, L, M, d_h,
            scale, lo_shift, static_cast<float*>(out), st);
    }
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int txl_attn_fwd(const void* q, const void* k, const void* v, const void* r_k,
                 const void* u_bias, const void* v_bias, int B, int H, int L, int M, int d_h,
                 float scale, void* out, int dtype, void* stream) {
    const int rc = check_attn_args(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, out, dtype);
    if (rc != TXL_OK) return rc;
    return launch_attn(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, scale, out, dtype, nullptr,
                       stream);
}

int txl_attn_fwd_ex(const void* q, const void* k, const void* v, const void* r_k,
                    const void* u_bias, const void* v_bias, int B, int H, int L, int M, int d_h,
                    float scale, int same_length, int mem_len, void* out, int dtype, void* stream) {
    const int rc = check_attn_args(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, out, dtype);
    if (rc != TXL_OK) return rc;
    if (same_length && (mem_len < M || mem_len >= (1 << 30))) return TXL_ERR_INVALID_ARG;
    return launch_attn(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, scale, out, dtype, nullptr,
                       stream, lower_shift(same_length, L, M, mem_len));
}

int txl_attn_bwd(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                 const void* v_bias, const void* dout, int B, int H, int L, int M, int d_h, float scale,
                 int same_length, int mem_len, float* dq, float* dk, float* dv, float* dr, float* du,
                 float* dvb, int dtype, void* stream) {
    const int rc = check_bwd_args(q, k, v, r_k, u_bias, v_bias, dout, B, H, L, M, d_h, same_length, mem_len, dq,
                                  dk, dv, dr, du, dvb, dtype);
    if (rc != TXL_OK) return rc;
    const cudaError_t e = txl::launch_attn_bwd_simt(q, k, v, r_k, u_bias, v_bias, dout, dtype == TXL_BF16, B, H,
                                                    L, M, d_h, scale, lower_shift(same_length, L, M, mem_len),
                                                    dq, dk, dv, dr, du, dvb, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

size_t txl_attn_bwd_workspace_bytes(int B, int H, int L, int M, int d_h, int dtype, int same_length) {
    // the tensor-core backward: bf16, d_h = 64, plain causal mask with memory
    if (dtype != TXL_BF16 || d_h != 64 || same_length || B <= 0 || H <= 0 || L <= 0 || M < 0) return 0;
    if ((long long)M + L >= (1ll << 30) || (long long)B * H >= (1ll << 30)) return 0;
    return txl::attn_bwd_tc_workspace_bytes(B, H, L, M);
}

int txl_attn_bwd_ws(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                    const void* v_bias, const void* dout, int B, int H, int L, int M, int d_h, float scale,
                    int same_length, int mem_len, float* dq, float* dk, float* dv, float* dr, float* du,
                    float* dvb, int dtype, void* workspace, size_t ws_bytes, void* stream) {
    const int rc = check_bwd_args(q, k, v, r_k, u_bias, v_bias, dout, B, H, L, M, d_h, same_length, mem_len, dq,
                                  dk, dv, dr, du, dvb, dtype);
    if (rc != TXL_OK) return rc;
    const size_t need = txl_attn_bwd_workspace_bytes(B, H, L, M, d_h, dtype, same_length);
    if (!need)
        return txl_attn_bwd(q, k, v, r_k, u_bias, v_bias, dout, B, H, L, M, d_h, scale, same_length, mem_len, dq,
                            dk, dv, dr, du, dvb, dtype, stream);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < need) return TXL_ERR_WORKSPACE;
    const long long K = (long long)M + L;
    const size_t nq = (size_t)B * H * L * d_h, nkv = (size_t)B * H * K * d_h, nr = (size_t)K * H * d_h,
                 nb = (size_t)H * d_h;
    const void* others[13] = {q, k, v, r_k, u_bias, v_bias, dout, dq, dk, dv, dr, du, dvb};
    const size_t sizes[13] = {nq * 2, nkv * 2, nkv * 2, nr * 2, nb * 2, nb * 2, nq * 2,
                              nq * 4, nkv * 4, nkv * 4, nr * 4, nb * 4, nb * 4};
    for (int o = 0; o < 13; ++o)
        if (overlap(workspace, need, others[o], sizes[o])) return TXL_ERR_ALIAS;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    const cudaError_t e =
        txl::launch_attn_bwd_tc(q, k, v, r_k, u_bias, v_bias, nullptr, nullptr, dout, B, H, L, M, scale, dq, dk, dv,
                                dr, du, dvb, workspace, status, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return TXL_ERR_CUDA;  // tensor-map encoding failed
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

int txl_attn_fwd_lse(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                     const void* v_bias, int B, int H, int L, int M, int d_h, float scale, void* out, float* lse,
                     int dtype, void* stream) {
    const int rc = check_attn_args(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, out, dtype);
    if (rc != TXL_OK) return rc;
    if (dtype != TXL_BF16) return TXL_ERR_UNSUPPORTED;
    if (!lse) return TXL_ERR_INVALID_ARG;
    if (!aligned16(lse)) return TXL_ERR_MISALIGNED;
    const size_t nl = (size_t)B * H * L * sizeof(float), nq = (size_t)B * H * L * d_h * 2,
                 nkv = (size_t)B * H * ((size_t)M + L) * d_h * 2, nr = ((size_t)M + L) * H * d_h * 2,
                 nb = (size_t)H * d_h * 2;
    if (overlap(lse, nl, out, nq) || overlap(lse, nl, q, nq) || overlap(lse, nl, k, nkv) ||
        overlap(lse, nl, v, nkv) || overlap(lse, nl, r_k, nr) || overlap(lse, nl, u_bias, nb) ||
        overlap(lse, nl, v_bias, nb))
        return TXL_ERR_ALIAS;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    g_inject = 0;
    const cudaError_t e = txl::launch_attn_tc_bf16_lse(q, k, v, r_k, u_bias, v_bias, B, H, L, M, scale,
                                                       kNoLowerBound, out, lse, status,
                                                       static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return TXL_ERR_CUDA;
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

int txl_attn_bwd_saved(const void* q, const void* k, const void* v, const void* r_k, const void* u_bias,
                       const void* v_bias, const void* out, const float* lse, const void* dout, int B, int H, int L,
                       int M, int d_h, float scale, float* dq, float* dk, float* dv, float* dr, float* du,
                       float* dvb, int dtype, void* workspace, size_t ws_bytes, void* stream) {
    const int rc = check_bwd_args(q, k, v, r_k, u_bias, v_bias, dout, B, H, L, M, d_h, 0, M, dq, dk, dv, dr, du,
                                  dvb, dtype);
    if (rc != TXL_OK) return rc;
    if (dtype != TXL_BF16 || d_h != 64) return TXL_ERR_UNSUPPORTED;
    if (!out || !lse) return TXL_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(lse)) return TXL_ERR_MISALIGNED;
    const size_t need = txl_attn_bwd_workspace_bytes(B, H, L, M, d_h, dtype, 0);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < need) return TXL_ERR_WORKSPACE;
    const long long K = (long long)M + L;
    const size_t nq = (size_t)B * H * L * d_h, nkv = (size_t)B * H * K * d_h, nr = (size_t)K * H * d_h,
                 nb = (size_t)H * d_h, nl = (size_t)B * H * L;
    const void* others[15] = {q, k, v, r_k, u_bias, v_bias, dout, out, lse, dq, dk, dv, dr, du, dvb};
    const size_t sizes[15] = {nq * 2, nkv * 2, nkv * 2, nr * 2, nb * 2, nb * 2, nq * 2, nq * 2, nl * 4,
                              nq * 4, nkv * 4, nkv * 4, nr * 4, nb * 4, nb * 4};
    for (int o = 0; o < 15; ++o)
        if (overlap(workspace, need, others[o], sizes[o])) return TXL_ERR_ALIAS;
    // the gradients must not overlap the saved forward state either
    const void* gr[6] = {dq, dk, dv, dr, du, dvb};
    const size_t gn[6] = {nq * 4, nkv * 4, nkv * 4, nr * 4, nb * 4, nb * 4};
    for (int o = 0; o < 6; ++o)
        if (overlap(gr[o], gn[o], out, nq * 2) || overlap(gr[o], gn[o], lse, nl * 4)) return TXL_ERR_ALIAS;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    const cudaError_t e =
        txl::launch_attn_bwd_tc(q, k, v, r_k, u_bias, v_bias, out, lse, dout, B, H, L, M, scale, dq, dk, dv, dr, du,
                                dvb, workspace, status, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return TXL_ERR_CUDA;
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

size_t txl_attn_workspace_bytes(int B, int H, int L, int M, int d_h, int dtype) {
    // only the bf16 kernel splits; sizes a call would reject need nothing
    if (dtype != TXL_BF16 || d_h != 64 || B <= 0 || H <= 0 || L <= 0 || M < 0) return 0;
    if ((long long)M + L >= (1ll << 30) || (long long)B * H >= (1ll << 30)) return 0;
    return txl::attn_tc_bf16_workspace_bytes(B, H, L, M);
}

int txl_attn_fwd_ws(const void* q, const void* k, const void* v, const void* r_k,
                    const void* u_bias, const void* v_bias, int B, int H, int L, int M, int d_h,
                    float scale, void* out, int dtype, void* workspace, size_t ws_bytes,
                    void* stream) {
    const int rc = check_attn_args(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, out, dtype);
    if (rc != TXL_OK) return rc;
    const size_t need = txl_attn_workspace_bytes(B, H, L, M, d_h, dtype);
    if (need) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < need)
            return TXL_ERR_WORKSPACE;
        const int es = elem_size(dtype);
        const size_t nq = (size_t)B * H * L * d_h * es, nkv = (size_t)B * H * ((size_t)M + L) * d_h * es;
        if (overlap(workspace, need, out, nq) || overlap(workspace, need, q, nq) ||
            overlap(workspace, need, k, nkv) || overlap(workspace, need, v, nkv))
            return TXL_ERR_ALIAS;
    }
    return launch_attn(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, scale, out, dtype,
                       need ? workspace : nullptr, stream);
}

int txl_mem_update(void* mems, const void* hids, int B, int L, int M, int d, int dtype,
                   void* stream) {
    return txl_mem_update_ext(mems, hids, B, L, M, d, 0, dtype, stream);
}

int txl_mem_update_ext(void* mems, const void* hids, int B, int L, int M, int d, int ext_len,
                       int dtype, void* stream) {
    const int es = elem_size(dtype);
    if (!es || B <= 0 || L <= 0 || M < 0 || d <= 0 || ext_len < 0) return TXL_ERR_INVALID_ARG;
    if (M == 0) return TXL_OK;
    if (!mems || !hids) return TXL_ERR_INVALID_ARG;
    if ((long long)B * (M > L ? M : L) * d >= (1ll << 40)) return TXL_ERR_UNSUPPORTED;
    const size_t row = (size_t)d * es;
    if (overlap(mems, (size_t)B * M * row, hids, (size_t)B * L * row)) return TXL_ERR_ALIAS;
    const int used = ext_len < L ? L - ext_len : 0;  // rows of h that enter the memory
    const cudaError_t e =
        txl::launch_tail_m(mems, hids, B, used, L, M, row, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

int txl_mem_ring_push(void* ring, const void* hids, int B, int L, int M, int d, int start,
                      int* new_start, int dtype, void* stream) {
    const int es = elem_size(dtype);
    if (!es || B <= 0 || L <= 0 || M < 0 || d <= 0 || !new_start) return TXL_ERR_INVALID_ARG;
    if (start < 0 || (M > 0 && start >= M) || (M == 0 && start != 0)) return TXL_ERR_INVALID_ARG;
    if (M == 0) {
        *new_start = 0;
        return TXL_OK;
    }
    if (!ring || !hids) return TXL_ERR_INVALID_ARG;
    if ((long long)B * (M > L ? M : L) * d >= (1ll << 40)) return TXL_ERR_UNSUPPORTED;
    const size_t row = (size_t)d * es;
    if (overlap(ring, (size_t)B * M * row, hids, (size_t)B * L * row)) return TXL_ERR_ALIAS;
    cudaError_t e;
    if (L >= M) {
        // the whole memory is replaced by the newest M rows: the Tail_M copy
        e = txl::launch_tail_m(ring, hids, B, L, L, M, row, static_cast<cudaStream_t>(stream));
        *new_start = 0;
    } else {
        e = txl::launch_ring_push(ring, hids, B, L, M, start, row, static_cast<cudaStream_t>(stream));
        *new_start = (start + L) % M;
    }
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

int txl_mem_reset(void* mems, const void* flags, int B, int rows, int d, int dtype, void* stream) {
    const int es = elem_size(dtype);
    if (!es || B <= 0 || rows < 0 || d <= 0 || !flags) return TXL_ERR_INVALID_ARG;
    if (rows == 0) return TXL_OK;
    if (!mems) return TXL_ERR_INVALID_ARG;
    const long long per_b = (long long)rows * d * es;
    if ((long long)B * per_b >= (1ll << 40)) return TXL_ERR_UNSUPPORTED;
    if (overlap(mems, (size_t)(B * per_b), flags, (size_t)B)) return TXL_ERR_ALIAS;
    const cudaError_t e = txl::launch_mem_reset(mems, static_cast<const unsigned char*>(flags), B, per_b,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

int txl_sync_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return TXL_ERR_CUDA;
    int status = 0;
    e = cudaMemcpyFromSymbol(&status, txl::g_dev_status, sizeof(int));
    if (e != cudaSuccess) return TXL_ERR_CUDA;
    if (status != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(txl::g_dev_status, &zero, sizeof(int)) != cudaSuccess)
            return TXL_ERR_CUDA;
        return TXL_ERR_DEVICE_TIMEOUT;
    }
    return TXL_OK;
}

int txl_attn_fwd_noalloc(const void* q, const void* k, const void* v, const void* r_k,
                         const void* u_bias, const void* v_bias, int B, int H, int L, int M,
                         int d_h, float scale, void* out, int dtype, void* stream) {
    const int rc = check_attn_args(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, out, dtype);
    if (rc != TXL_OK) return rc;
    const size_t need = txl_attn_workspace_bytes(B, H, L, M, d_h, dtype);
    if (need > TXL_NOALLOC_SCRATCH_BYTES) return TXL_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (need) {
        scratch = noalloc_scratch(static_cast<cudaStream_t>(stream));
        if (!scratch) return TXL_ERR_CUDA;
    }
    return launch_attn(q, k, v, r_k, u_bias, v_bias, B, H, L, M, d_h, scale, out, dtype, scratch,
                       stream);
}

int txl_qkv_proj(const void* h, const void* mem, const void* w_qkv, int B, int L, int M, int H,
                 int d_h, void* q, void* k, void* v, void* stream) {
    return txl_qkv_proj_ex(h, TXL_LAYOUT_ROWS, mem, TXL_LAYOUT_ROWS, w_qkv, B, L, M, H, d_h, q, k, v,
                           stream);
}

int txl_qkv_proj_ex(const void* h, int h_layout, const void* mem, int mem_layout,
                    const void* w_qkv, int B, int L, int M, int H, int d_h, void* q, void* k,
                    void* v, void* stream) {
    return txl_qkv_proj_ring(h, h_layout, mem, mem_layout, 0, w_qkv, B, L, M, H, d_h, q, k, v, stream);
}

}  // extern "C"

namespace {

// Host validation of the q/k/v projections (txl_qkv_proj_ring's contract).
int check_qkv(const void* h, int h_layout, const void* mem, int mem_layout, int mem_start,
              const void* w_qkv, int B, int L, int M, int H, int d_h, void* q, void* k, void* v) {
    if (!h || !w_qkv || !q || !k || !v || (M > 0 && !mem)) return TXL_ERR_INVALID_ARG;
    const auto layout_ok = [](int l) { return l == TXL_LAYOUT_ROWS || l == TXL_LAYOUT_HEADS; };
    if (!layout_ok(h_layout) || !layout_ok(mem_layout)) return TXL_ERR_INVALID_ARG;
    if (mem_start < 0 || (M > 0 && mem_start >= M) || (M == 0 && mem_start != 0))
        return TXL_ERR_INVALID_ARG;
    if (mem_start % 128 != 0) return TXL_ERR_UNSUPPORTED;
    if (B <= 0 || L <= 0 || M < 0 || H <= 0 || d_h <= 0) return TXL_ERR_INVALID_ARG;
    if (d_h != 64 || H % 4 != 0 || L % 128 != 0 || M % 128 != 0) return TXL_ERR_UNSUPPORTED;
    const long long d = (long long)H * d_h;
    if ((long long)B * (M + L) * d >= (1ll << 31) || (long long)(M + L) >= (1ll << 20))
        return TXL_ERR_UNSUPPORTED;
    if (!aligned16(h) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        (M > 0 && !aligned16(mem)))
        return TXL_ERR_MISALIGNED;
    const size_t nh = (size_t)B * L * d * 2, nm = (size_t)B * M * d * 2, nw = (size_t)3 * d * d * 2;
    const size_t nq = nh, nkv = (size_t)B * (M + L) * d * 2;
    const void* outs[3] = {q, k, v};
    const size_t nout[3] = {nq, nkv, nkv};
    for (int o = 0; o < 3; ++o) {
        if (overlap(outs[o], nout[o], h, nh) || overlap(outs[o], nout[o], w_qkv, nw) ||
            (M > 0 && overlap(outs[o], nout[o], mem, nm)))
            return TXL_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlap(outs[o], nout[o], outs[o2], nout[o2])) return TXL_ERR_ALIAS;
    }
    return TXL_OK;
}

// Host validation of the position projection (txl_r_proj's contract).
int check_r(const void* emb, const void* w_r, int K, int H, int d_h, void* r_k) {
    if (!emb || !w_r || !r_k || K <= 0 || H <= 0 || d_h <= 0) return TXL_ERR_INVALID_ARG;
    if (d_h != 64 || H % 4 != 0 || K % 128 != 0) return TXL_ERR_UNSUPPORTED;
    const long long d = (long long)H * d_h;
    if ((long long)K * d >= (1ll << 31)) return TXL_ERR_UNSUPPORTED;
    if (!aligned16(emb) || !aligned16(w_r) || !aligned16(r_k)) return TXL_ERR_MISALIGNED;
    const size_t nr = (size_t)K * d * 2;
    if (overlap(r_k, nr, emb, nr) || overlap(r_k, nr, w_r, (size_t)d * d * 2)) return TXL_ERR_ALIAS;
    return TXL_OK;
}

// The q and k|v problems of one layer's projection launch.
void qkv_problems(txl::ProjGemm* gm, const void* h, int h_layout, const void* mem, int mem_layout,
                  int mem_start, const void* w_qkv, int L, int M, long long d, void* q, void* k, void* v) {
    const unsigned char* w = static_cast<const unsigned char*>(w_qkv);
    const int hh = h_layout == TXL_LAYOUT_HEADS, mh = mem_layout == TXL_LAYOUT_HEADS;
    gm[0] = {nullptr, h, 0, L, 0, hh, w, (int)d, L, {q, nullptr, nullptr}};
    gm[1] = {M > 0 ? mem : nullptr, h, M, L, mh, hh, w + (size_t)d * d * 2, (int)(2 * d), M + L,
             {k, v, nullptr}, mem_start};
}

int launch_status(cudaError_t e) {
    if (e == cudaErrorInvalidValue) return TXL_ERR_CUDA;  // a tensor map could not be encoded
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int txl_qkv_proj_ring(const void* h, int h_layout, const void* mem, int mem_layout, int mem_start,
                      const void* w_qkv, int B, int L, int M, int H, int d_h, void* q, void* k,
                      void* v, void* stream) {
    const int rc = check_qkv(h, h_layout, mem, mem_layout, mem_start, w_qkv, B, L, M, H, d_h, q, k, v);
    if (rc != TXL_OK) return rc;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    // one launch: q from h and W_q; k, v from [mem; h] and the W_k, W_v rows
    txl::ProjGemm gm[2];
    qkv_problems(gm, h, h_layout, mem, mem_layout, mem_start, w_qkv, L, M, (long long)H * d_h, q, k, v);
    return launch_status(txl::launch_proj_gemm(gm, 2, B, H * d_h, H * d_h, H, d_h, 0, status,
                                               static_cast<cudaStream_t>(stream)));
}

int txl_qkvr_proj(const void* h, int h_layout, const void* mem, int mem_layout, int mem_start,
                  const void* w_qkv, const void* emb, const void* w_r, int B, int L, int M, int H,
                  int d_h, void* q, void* k, void* v, void* r_k, void* stream) {
    int rc = check_qkv(h, h_layout, mem, mem_layout, mem_start, w_qkv, B, L, M, H, d_h, q, k, v);
    if (rc != TXL_OK) return rc;
    rc = check_r(emb, w_r, M + L, H, d_h, r_k);
    if (rc != TXL_OK) return rc;
    const long long d = (long long)H * d_h;
    const size_t nr = (size_t)(M + L) * d * 2, nq = (size_t)B * L * d * 2, nkv = (size_t)B * (M + L) * d * 2;
    const size_t nh = nq, nm = (size_t)B * M * d * 2, nw = (size_t)3 * d * d * 2;
    // r_k overlaps no other output and no input of the q/k/v problems
    if (overlap(r_k, nr, q, nq) || overlap(r_k, nr, k, nkv) || overlap(r_k, nr, v, nkv) ||
        overlap(r_k, nr, h, nh) || overlap(r_k, nr, w_qkv, nw) || (M > 0 && overlap(r_k, nr, mem, nm)))
        return TXL_ERR_ALIAS;
    const void* outs[3] = {q, k, v};
    const size_t nout[3] = {nq, nkv, nkv};
    for (int o = 0; o < 3; ++o)
        if (overlap(outs[o], nout[o], emb, nr) || overlap(outs[o], nout[o], w_r, (size_t)d * d * 2))
            return TXL_ERR_ALIAS;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    // one launch: q, k|v as in txl_qkv_proj_ring, and r from the position
    // embedding (one batch row, row-major output)
    txl::ProjGemm gm[3];
    qkv_problems(gm, h, h_layout, mem, mem_layout, mem_start, w_qkv, L, M, d, q, k, v);
    gm[2] = {nullptr, emb, 0, M + L, 0, 0, w_r, (int)d, M + L, {r_k, nullptr, nullptr}, 0, 1, 1};
    return launch_status(txl::launch_proj_gemm(gm, 3, B, (int)d, (int)d, H, d_h, 0, status,
                                               static_cast<cudaStream_t>(stream)));
}

int txl_r_proj(const void* emb, const void* w_r, int K, int H, int d_h, void* r_k, void* stream) {
    const int rc = check_r(emb, w_r, K, H, d_h, r_k);
    if (rc != TXL_OK) return rc;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    const long long d = (long long)H * d_h;
    const txl::ProjGemm gm = {nullptr, emb, 0, K, 0, 0, w_r, (int)d, K, {r_k, nullptr, nullptr}};
    return launch_status(txl::launch_proj_gemm(&gm, 1, 1, (int)d, (int)d, H, d_h, 1, status,
                                               static_cast<cudaStream_t>(stream)));
}

int txl_linear(const void* x, int x_layout, int B, int T, int K, const void* w, int N,
               const void* bias, const void* resid, int relu, void* out, void* stream) {
    if (!x || !w || !out || B <= 0 || T <= 0 || K <= 0 || N <= 0) return TXL_ERR_INVALID_ARG;
    if (x_layout != TXL_LAYOUT_ROWS && x_layout != TXL_LAYOUT_HEADS) return TXL_ERR_INVALID_ARG;
    if (T % 128 != 0 || K % 64 != 0 || N % 256 != 0) return TXL_ERR_UNSUPPORTED;
    if ((long long)B * T * (K > N ? K : N) >= (1ll << 31) || (long long)T >= (1ll << 24))
        return TXL_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (bias && !aligned16(bias)) ||
        (resid && !aligned16(resid)))
        return TXL_ERR_MISALIGNED;
    const size_t nx = (size_t)B * T * K * 2, nw = (size_t)N * K * 2, no = (size_t)B * T * N * 2;
    if (overlap(out, no, x, nx) || overlap(out, no, w, nw) || (bias && overlap(out, no, bias, (size_t)N * 2)))
        return TXL_ERR_ALIAS;
    if (resid && resid != out && overlap(out, no, resid, no)) return TXL_ERR_ALIAS;
    int* status = dev_status_ptr();
    if (!status) return TXL_ERR_CUDA;
    const cudaError_t e = txl::launch_linear(x, x_layout == TXL_LAYOUT_HEADS, B, T, K, w, N, bias, resid,
                                             relu ? 1 : 0, out, status, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return TXL_ERR_CUDA;
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

int txl_layer_norm(const void* x, const void* y, const void* gamma, const void* beta, long long rows,
                   int d, float eps, void* out, void* stream) {
    if (!x || !gamma || !beta || !out || rows < 0 || d <= 0 || !(eps >= 0.f)) return TXL_ERR_INVALID_ARG;
    if (d % 256 != 0 || d > 2048 || d == 1280 || d == 1792) return TXL_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) || (y && !aligned16(y)))
        return TXL_ERR_MISALIGNED;
    const size_t n = (size_t)rows * d * 2;
    if ((out != x && overlap(out, n, x, n)) || (y && out != y && overlap(out, n, y, n)) ||
        overlap(out, n, gamma, (size_t)d * 2) || overlap(out, n, beta, (size_t)d * 2))
        return TXL_ERR_ALIAS;
    const cudaError_t e =
        txl::launch_layer_norm(x, y, gamma, beta, rows, d, eps, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TXL_OK : TXL_ERR_LAUNCH;
}

const char* txl_status_string(int status) {
    switch (status) {
        case TXL_OK: return "ok";
        case TXL_ERR_INVALID_ARG: return "invalid argument";
        case TXL_ERR_UNSUPPORTED: return "unsupported size";
        case TXL_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case TXL_ERR_ALIAS: return "output overlaps an input";
        case TXL_ERR_LAUNCH: return "kernel launch failed";
        case TXL_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case TXL_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case TXL_ERR_CUDA: return "CUDA runtime/driver call failed";
        case TXL_ERR_SCRATCH_LIMIT: return "call needs more scratch than the static no-alloc buffer";
        case TXL_ERR_OUT_OF_BOUNDS: return "a bounds-checked kernel skipped an out-of-range access";
        default: return "unknown status";
    }
}

int txl_version(void) { return (1 << 16) | 0; }

int txl_bounds_status(unsigned long long* first) {
#ifndef TXL_CHECKED
    if (first) *first = 0;
    return TXL_ERR_UNSUPPORTED;  // this library was built without bounds checks
#else
    if (cudaDeviceSynchronize() != cudaSuccess) return TXL_ERR_CUDA;
    const unsigned long long words[7] = {txl::bounds_word_attn_simt(),   txl::bounds_word_attn_tc(),
                                         txl::bounds_word_attn_bwd(),    txl::bounds_word_attn_bwd_tc(),
                                         txl::bounds_word_mem_update(),  txl::bounds_word_layer_norm(),
                                         txl::bounds_word_proj_gemm()};
    unsigned long long w = 0;
    for (unsigned long long x : words) {
        if (x == ~0ull) return TXL_ERR_CUDA;
        if (!w && x) w = x;
    }
    if (first) *first = w;
    return w ? TXL_ERR_OUT_OF_BOUNDS : TXL_OK;
#endif
}

int txl_debug_inject(int kind) {
    if (kind < 0 || kind > 1) return TXL_ERR_INVALID_ARG;
    g_inject = kind;
    return TXL_OK;
}

}  // extern "C"
