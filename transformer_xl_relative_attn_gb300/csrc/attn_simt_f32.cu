// fp32 relative attention on CUDA cores (the TXL_F32 path).
//
// One warp owns one query row i of one (batch row, head).  Keys are swept in
// chunks of 32, one key per lane, with an online softmax: each lane forms
//   s(i,j) = scale * ((q_i+u).k_j + (q_i+v).R[M+L-1-(M+i-j)])
// for its key ("Transformer-XL模型 核心源码阅读笔记", section "Build the
// model", RelPartialLearnableMultiHeadAttn.forward: AC + BD after the shift),
// keys past M+i are masked ("Transformer-XL" notes, section "Causal Mask With
// Memory"; with same_length also keys before i+1-lo_shift, per the source
// notes' MemTransformerLM._forward), and the chunk's probabilities are broadcast lane by lane while
// each lane accumulates its own output columns.  The relative shift is the
// row index M+L-1-(M+i-j) of R; no shifted score matrix is formed.
#include <cstdint>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

constexpr int kSimtMaxD = 256;
constexpr int kSimtWarps = 4;

__global__ void __launch_bounds__(32 * kSimtWarps)
attn_simt_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                     const float* __restrict__ v, const float* __restrict__ r,
                     const float* __restrict__ ub, const float* __restrict__ vb, int B, int H,
                     int L, int M, int dh, float scale, int lo_shift, float* __restrict__ out) {
    __shared__ float s_qu[kSimtWarps][kSimtMaxD];
    __shared__ float s_qv[kSimtWarps][kSimtMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kSimtWarps + warp;
    if (row >= (long long)B * H * L) return;
    const int i = (int)(row % L);
    const long long bh = row / L;
    const int h = (int)(bh % H);
    const int K = M + L;
    const float* qi = q + row * dh;
    const long long n_q = (long long)B * H * L * dh, n_kv = (long long)B * H * K * dh;
    const long long n_r = (long long)K * H * dh, n_b = (long long)H * dh;
    for (int t = lane; t < dh; t += 32) {
        const float x = TXL_BOUNDS(row * dh + t < n_q, 101, row * dh + t) ? qi[t] : 0.f;
        const bool bo = TXL_BOUNDS(h * dh + t < n_b, 102, h * dh + t);
        s_qu[warp][t] = x + (bo ? ub[h * dh + t] : 0.f);
        s_qv[warp][t] = x + (bo ? vb[h * dh + t] : 0.f);
    }
    __syncwarp();
    const float* kb = k + bh * (long long)K * dh;
    const float* vbase = v + bh * (long long)K * dh;
    const int nvis = M + i + 1;  // keys up to M+i are visible
    const int jlo = max(0, i + 1 - lo_shift);  // ... from jlo on (0 unless same_length)
    const int ncol = (dh + 31) / 32;
    float acc[kSimtMaxD / 32];
#pragma unroll
    for (int c = 0; c < kSimtMaxD / 32; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int j0 = jlo; j0 < nvis; j0 += 32) {
        const int j = j0 + lane;
        float s = -INFINITY;
        if (j < nvis) {
            const int dist = M + i - j;
            const float* kj = kb + (long long)j * dh;
            const long long ri = ((long long)(K - 1 - dist) * H + h) * dh;
            const float* rj = r + ri;
            float ac = 0.f, bd = 0.f;
            const bool kin = TXL_BOUNDS((bh * K + j) * dh + dh <= n_kv, 103, (bh * K + j) * dh);
            const bool rin = TXL_BOUNDS(ri >= 0 && ri + dh <= n_r, 104, ri);
            for (int t = 0; t < dh; ++t) {
                if (kin) ac = fmaf(s_qu[warp][t], kj[t], ac);
                if (rin) bd = fmaf(s_qv[warp][t], rj[t], bd);
            }
            s = scale * (ac + bd);
        }
        float cm = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        const float mn = fmaxf(m, cm);
        const float alpha = expf(m - mn);  // 0 on the first chunk (m = -inf)
        const float p = (j < nvis) ? expf(s - mn) : 0.f;
        float ps = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l = l * alpha + ps;
        m = mn;
#pragma unroll
        for (int c = 0; c < kSimtMaxD / 32; ++c) acc[c] *= alpha;
        const int nk = min(32, nvis - j0);
        for (int jj = 0; jj < nk; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const float* vj = vbase + (long long)(j0 + jj) * dh;
            if (!TXL_BOUNDS((bh * K + j0 + jj) * dh + dh <= n_kv, 105, (bh * K + j0 + jj) * dh)) continue;
#pragma unroll
            for (int c = 0; c < kSimtMaxD / 32; ++c) {
                const int t = lane + 32 * c;
                if (c < ncol && t < dh) acc[c] = fmaf(pj, vj[t], acc[c]);
            }
        }
    }
    const float inv = 1.f / l;
    float* o = out + row * dh;
#pragma unroll
    for (int c = 0; c < kSimtMaxD / 32; ++c) {
        const int t = lane + 32 * c;
        if (c < ncol && t < dh && TXL_BOUNDS(row * dh + t < n_q, 106, row * dh + t)) o[t] = acc[c] * inv;
    }
}

cudaError_t launch_attn_simt_f32(const float* q, const float* k, const float* v, const float* r,
                                 const float* ub, const float* vb, int B, int H, int L, int M,
                                 int dh, float scale, int lo_shift, float* out, cudaStream_t stream) {
    const long long rows = (long long)B * H * L;
    const long long blocks = (rows + kSimtWarps - 1) / kSimtWarps;
    if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    attn_simt_f32_kernel<<<(unsigned)blocks, 32 * kSimtWarps, 0, stream>>>(
        q, k, v, r, ub, vb, B, H, L, M, dh, scale, lo_shift, out);
    return cudaGetLastError();
}

TXL_BOUNDS_READER(bounds_word_attn_simt)

}  // namespace txl
