// Backward of the relative attention on CUDA cores (fp32 arithmetic, inputs
// fp32 or bf16, gradients fp32), for training with a stop-gradient memory
// ("Transformer-XL" notes, zty624: the memory is a constant input of the
// segment, so nothing flows into the previous segment; the memory rows'
// keys and values still get their gradients, which the caller drops).
//
// From the forward s_ij = scale ((q_i+u).k_j + (q_i+v).R[K-1-(M+i-j)]),
// P = softmax_j(s), O_i = sum_j P_ij V_j, and dO:
//   dP_ij = dO_i . V_j,   D_i = sum_j P_ij dP_ij  (= dO_i . O_i),
//   dS_ij = P_ij (dP_ij - D_i)
//   dq_i = scale sum_j dS_ij (k_j + R_ij),  dk_j += scale dS_ij (q_i + u),
//   dV_j += P_ij dO_i,  dR_row += scale dS_ij (q_i + v),
//   du += scale sum_j dS_ij k_j,  dv += scale sum_j dS_ij R_ij.
//
// One warp owns one query row of one (batch row, head) and sweeps its
// visible keys three times, one key per lane: (1) row max and sum of exp,
// (2) D_i, (3) dS, with the per-key contributions broadcast lane by lane
// while each lane owns output columns lane, lane+32, ...  dq is written once;
// dk, dV, dR, du and dv are summed over query rows with fp32 atomics into
// buffers the host zeroes first.  A correctness path: its cost is the
// atomics, not the arithmetic.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include "txl_device.cuh"

namespace txl {

constexpr int kBwdMaxD = 256;
constexpr int kBwdWarps = 4;

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Element idx of an array of n elements (bounds-checked builds skip and
// record an index outside it; otherwise the check compiles away).
template <typename T>
__device__ __forceinline__ float ld_at(const T* base, long long idx, long long n, int site) {
    return TXL_BOUNDS(idx >= 0 && idx < n, site, idx) ? ld_f(base + idx) : 0.f;
}
__device__ __forceinline__ void add_at(float* base, long long idx, long long n, int site, float v) {
    if (TXL_BOUNDS(idx >= 0 && idx < n, site, idx)) atomicAdd(base + idx, v);
}

template <typename T>
__global__ void __launch_bounds__(32 * kBwdWarps)
attn_bwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ r, const T* __restrict__ ub, const T* __restrict__ vb,
                     const T* __restrict__ dout, int B, int H, int L, int M, int dh, float scale,
                     int lo_shift, float* __restrict__ dq, float* __restrict__ dk,
                     float* __restrict__ dv, float* __restrict__ dr, float* __restrict__ du,
                     float* __restrict__ dvb) {
    __shared__ float s_qu[kBwdWarps][kBwdMaxD];
    __shared__ float s_qv[kBwdWarps][kBwdMaxD];
    __shared__ float s_do[kBwdWarps][kBwdMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kBwdWarps + warp;
    if (row >= (long long)B * H * L) return;
    const int i = (int)(row % L);
    const long long bh = row / L;
    const int h = (int)(bh % H);
    const int K = M + L;
    const long long n_q = (long long)B * H * L * dh, n_kv = (long long)B * H * K * dh;
    const long long n_r = (long long)K * H * dh, n_b = (long long)H * dh;
    for (int t = lane; t < dh; t += 32) {
        const float x = ld_at(q, row * dh + t, n_q, 501);
        s_qu[warp][t] = x + ld_at(ub, (long long)h * dh + t, n_b, 502);
        s_qv[warp][t] = x + ld_at(vb, (long long)h * dh + t, n_b, 503);
        s_do[warp][t] = ld_at(dout, row * dh + t, n_q, 504);
    }
    __syncwarp();
    const int nvis = M + i + 1;                   // keys up to M+i
    const int jlo = max(0, i + 1 - lo_shift);     // ... from jlo on (same_length)
    const int ncol = (dh + 31) / 32;

    auto score = [&](int j) {
        const int dist = M + i - j;
        const long long ki = (bh * K + j) * dh, ri = ((long long)(K - 1 - dist) * H + h) * dh;
        float ac = 0.f, bd = 0.f;
        for (int t = 0; t < dh; ++t) {
            ac = fmaf(s_qu[warp][t], ld_at(k, ki + t, n_kv, 505), ac);
            bd = fmaf(s_qv[warp][t], ld_at(r, ri + t, n_r, 506), bd);
        }
        return scale * (ac + bd);
    };
    auto dprob = [&](int j) {
        const long long vi = (bh * K + j) * dh;
        float a = 0.f;
        for (int t = 0; t < dh; ++t) a = fmaf(s_do[warp][t], ld_at(v, vi + t, n_kv, 507), a);
        return a;
    };

    // (1) row max and sum of exp
    float m = -INFINITY, l = 0.f;
    for (int j0 = jlo; j0 < nvis; j0 += 32) {
        const int j = j0 + lane;
        const float s = j < nvis ? score(j) : -INFINITY;
        float cm = s;
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        const float mn = fmaxf(m, cm);
        float e = j < nvis ? expf(s - mn) : 0.f;
        for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
        l = l * expf(m - mn) + e;
        m = mn;
    }
    const float inv_l = 1.f / l;
    // (2) D = sum_j P_ij dP_ij
    float D = 0.f;
    for (int j0 = jlo; j0 < nvis; j0 += 32) {
        const int j = j0 + lane;
        float c = 0.f;
        if (j < nvis) c = expf(score(j) - m) * inv_l * dprob(j);
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        D += c;
    }
    // (3) dS and the contributions
    float gq_c[kBwdMaxD / 32], gq_p[kBwdMaxD / 32];
#pragma unroll
    for (int c = 0; c < kBwdMaxD / 32; ++c) gq_c[c] = gq_p[c] = 0.f;
    for (int j0 = jlo; j0 < nvis; j0 += 32) {
        const int j = j0 + lane;
        float p = 0.f, ds = 0.f;
        if (j < nvis) {
            p = expf(score(j) - m) * inv_l;
            ds = p * (dprob(j) - D);
        }
        const int nk = min(32, nvis - j0);
        for (int jj = 0; jj < nk; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const float dsj = __shfl_sync(0xffffffffu, ds, jj);
            const int jk = j0 + jj;
            const long long rrow = (long long)(K - 1 - (M + i - jk));
            const long long kvi = (bh * K + jk) * dh, ri = (rrow * H + h) * dh;
#pragma unroll
            for (int c = 0; c < kBwdMaxD / 32; ++c) {
                const int t = lane + 32 * c;
                if (c < ncol && t < dh) {
                    gq_c[c] = fmaf(dsj, ld_at(k, kvi + t, n_kv, 508), gq_c[c]);
                    gq_p[c] = fmaf(dsj, ld_at(r, ri + t, n_r, 509), gq_p[c]);
                    add_at(dk, kvi + t, n_kv, 510, scale * dsj * s_qu[warp][t]);
                    add_at(dv, kvi + t, n_kv, 511, pj * s_do[warp][t]);
                    add_at(dr, ri + t, n_r, 512, scale * dsj * s_qv[warp][t]);
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kBwdMaxD / 32; ++c) {
        const int t = lane + 32 * c;
        if (c < ncol && t < dh) {
            if (TXL_BOUNDS(row * dh + t < n_q, 513, row * dh + t)) dq[row * dh + t] = scale * (gq_c[c] + gq_p[c]);
            add_at(du, (long long)h * dh + t, n_b, 514, scale * gq_c[c]);
            add_at(dvb, (long long)h * dh + t, n_b, 515, scale * gq_p[c]);
        }
    }
}


// Block-cooperative version for d_h <= 64: a CTA of 8 warps owns 32
// consecutive query rows of one (batch row, head), 4 per warp, and sweeps the
// keys any of them sees in chunks of 32.  Each chunk's K and V rows and the
// 63 R rows its 32 x 32 pairs use are staged in shared memory once for all
// 32 query rows; every product reads 16-byte vectors (staged rows padded to
// 68 floats, 17 vectors, so the 8 lanes of a quarter warp reading 8 keys'
// rows hit distinct banks).  Sweep 1 gives each row its max, its sum of exp and D_i (online),
// sweep 2 the chunk's P and dS tiles in shared memory, from which every
// contribution is a small product (dq per row in registers; dk, dV per key
// and dR per distance summed over the 32 rows), flushed to the global sums
// with one fp32 atomic per element per chunk.
constexpr int kQR = 32;         // query rows per CTA
constexpr int kRPW = 4;         // query rows per warp (8 warps)
constexpr int kDT = 64;         // d_h capacity
constexpr int kPad = 68;        // padded row of a staged tile (17 x 16 bytes)
constexpr int kSpan = 63;       // distances one 32 x 32 block of pairs covers
constexpr int kPS = 33;         // padded row of the P and dS tiles
constexpr size_t kTiledSmem =
    (size_t)(3 * kQR * kDT + 2 * kQR * kPad + kSpan * kPad + 2 * kQR * kPS) * sizeof(float);

// Three CTAs per SM (80 registers a thread, 28 bytes of spills; 3 x 66 KB of
// shared memory): one CTA's 8 warps alone left the SM waiting on
// shared-memory latency; base512 call 9.9 ms with one CTA, 8.6 with two,
// 8.25 with three.
template <typename T>
__global__ void __launch_bounds__(256, 3)
attn_bwd_tiled_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const T* __restrict__ r, const T* __restrict__ ub, const T* __restrict__ vb,
                      const T* __restrict__ dout, int B, int H, int L, int M, int dh, float scale,
                      int lo_shift, float* __restrict__ dq, float* __restrict__ dk,
                      float* __restrict__ dv, float* __restrict__ dr, float* __restrict__ du,
                      float* __restrict__ dvb) {
    extern __shared__ float sm[];
    float* s_qu = sm;                    // [32 rows][64]
    float* s_qv = s_qu + kQR * kDT;
    float* s_do = s_qv + kQR * kDT;
    float* t_k = s_do + kQR * kDT;       // [32 keys][65] of the chunk
    float* t_v = t_k + kQR * kPad;
    float* t_r = t_v + kQR * kPad;       // [63 slots][65]: slot = row - key + 31
    float* s_p = t_r + kSpan * kPad;     // [32 rows][33]: P of the chunk
    float* s_s = s_p + kQR * kPS;        // [32 rows][33]: dS of the chunk
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nqt = (L + kQR - 1) / kQR;
    const long long bh = blockIdx.x / nqt;
    const int i0 = (int)(blockIdx.x % nqt) * kQR;
    const int h = (int)(bh % H);
    const int K = M + L;
    const long long n_q = (long long)B * H * L * dh, n_kv = (long long)B * H * K * dh;
    const long long n_r = (long long)K * H * dh, n_b = (long long)H * dh;
    for (int idx = tid; idx < kQR * kDT; idx += 256) {
        const int rr = idx / kDT, t = idx % kDT, i = i0 + rr;
        float a = 0.f, b = 0.f, c = 0.f;
        if (i < L && t < dh) {
            const float x = ld_at(q, (bh * L + i) * dh + t, n_q, 521);
            a = x + ld_at(ub, (long long)h * dh + t, n_b, 522);
            b = x + ld_at(vb, (long long)h * dh + t, n_b, 523);
            c = ld_at(dout, (bh * L + i) * dh + t, n_q, 524);
        }
        s_qu[idx] = a;
        s_qv[idx] = b;
        s_do[idx] = c;
    }
    const int imax = min(i0 + kQR - 1, L - 1);
    const int jstart = max(0, i0 + 1 - lo_shift), jend = M + imax + 1;

    // stage the chunk at j0: K, V rows j0 .. j0+31 and the R row of each slot
    auto stage = [&](int j0) {
        __syncthreads();
        for (int idx = tid; idx < kQR * kDT; idx += 256) {
            const int jj = idx / kDT, t = idx % kDT, j = j0 + jj;
            float a = 0.f, b = 0.f;
            if (j < K && t < dh) {
                a = ld_at(k, (bh * K + j) * dh + t, n_kv, 525);
                b = ld_at(v, (bh * K + j) * dh + t, n_kv, 526);
            }
            t_k[jj * kPad + t] = a;
            t_v[jj * kPad + t] = b;
        }
        for (int idx = tid; idx < kSpan * kDT; idx += 256) {
            const int sl = idx / kDT, t = idx % kDT;
            const long long rrow = (long long)K - 1 - (M + (sl - 31) + i0 - j0);
            t_r[sl * kPad + t] = (rrow >= 0 && rrow < K && t < dh) ? ld_at(r, (rrow * H + h) * dh + t, n_r, 527) : 0.f;
        }
        __syncthreads();
    };
    // score of (row rr, key j0 + lane) from the staged tiles
    // 16-byte views (padding beyond d_h is zero, so whole vectors are summed)
    const float4* q4u = reinterpret_cast<const float4*>(s_qu);
    const float4* q4v = reinterpret_cast<const float4*>(s_qv);
    const float4* d4o = reinterpret_cast<const float4*>(s_do);
    const float4* k4 = reinterpret_cast<const float4*>(t_k);
    const float4* v4 = reinterpret_cast<const float4*>(t_v);
    const float4* r4 = reinterpret_cast<const float4*>(t_r);
    constexpr int RV = kDT / 4, TV = kPad / 4;  // vectors per row of the row tiles, staged tiles
    auto dot4 = [](float4 a, float4 b, float c) {
        return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, c))));
    };
    auto score = [&](int rr, int jj) {
        const int kb4 = jj * TV, rb4 = (rr - jj + 31) * TV;
        float ac = 0.f, bd = 0.f;
#pragma unroll
        for (int u = 0; u < RV; ++u) {
            ac = dot4(q4u[rr * RV + u], k4[kb4 + u], ac);
            bd = dot4(q4v[rr * RV + u], r4[rb4 + u], bd);
        }
        return scale * (ac + bd);
    };
    auto dprob = [&](int rr, int jj) {
        float a = 0.f;
#pragma unroll
        for (int u = 0; u < RV; ++u) a = dot4(d4o[rr * RV + u], v4[jj * TV + u], a);
        return a;
    };
    auto visible = [&](int i, int j) { return i < L && j < jend && j <= M + i && j >= i + 1 - lo_shift; };

    float m[kRPW], l[kRPW], D[kRPW];
#pragma unroll
    for (int w = 0; w < kRPW; ++w) {
        m[w] = -INFINITY;
        l[w] = 0.f;
        D[w] = 0.f;
    }
    // sweep 1: max, sum of exp and D = sum_j P dP, online (the sums are
    // rescaled whenever the running max grows; D is divided by l at the end)
    for (int j0 = jstart; j0 < jend; j0 += 32) {
        stage(j0);
#pragma unroll
        for (int w = 0; w < kRPW; ++w) {
            const int rr = warp * kRPW + w, i = i0 + rr, j = j0 + lane;
            const bool vis = visible(i, j);
            const float s = vis ? score(rr, lane) : -INFINITY;
            float cm = s;
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            const float mn = fmaxf(m[w], cm);
            if (mn == -INFINITY) continue;  // no visible key of this row yet
            const float e = vis ? expf(s - mn) : 0.f;
            float es = e, ed = vis ? e * dprob(rr, lane) : 0.f;
            for (int o = 16; o > 0; o >>= 1) {
                es += __shfl_xor_sync(0xffffffffu, es, o);
                ed += __shfl_xor_sync(0xffffffffu, ed, o);
            }
            const float a = expf(m[w] - mn);
            l[w] = l[w] * a + es;
            D[w] = D[w] * a + ed;
            m[w] = mn;
        }
    }
#pragma unroll
    for (int w = 0; w < kRPW; ++w)
        if (l[w] > 0.f) D[w] /= l[w];
    // sweep 2: P and dS of each chunk into shared tiles, then every
    // contribution as a small product over those tiles: thread (row or key
    // or distance slot = tid / 8, columns tid % 8 + 8c) with no shuffles and
    // no shared atomics; dk, dV, dR flushed with one global atomic each.
    const int rid = tid >> 3, cg = tid & 7;
    // thread columns: 4 cg .. 4 cg + 3 (vector cg) and 32 + 4 cg .. (vector 8 + cg)
    auto fma4 = [](float s, float4 a, float4& acc) {
        acc.x = fmaf(s, a.x, acc.x);
        acc.y = fmaf(s, a.y, acc.y);
        acc.z = fmaf(s, a.z, acc.z);
        acc.w = fmaf(s, a.w, acc.w);
    };
    float4 gc[2], gp[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) gc[c] = gp[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = jstart; j0 < jend; j0 += 32) {
        stage(j0);
#pragma unroll
        for (int w = 0; w < kRPW; ++w) {
            const int rr = warp * kRPW + w, i = i0 + rr, j = j0 + lane;
            float p = 0.f, ds = 0.f;
            if (visible(i, j)) {
                p = expf(score(rr, lane) - m[w]) / l[w];
                ds = p * (dprob(rr, lane) - D[w]);
            }
            s_p[rr * kPS + lane] = p;
            s_s[rr * kPS + lane] = ds;
        }
        __syncthreads();
        // dq of row rid: sum over the chunk's keys
        for (int jj = 0; jj < 32; ++jj) {
            const float dsv = s_s[rid * kPS + jj];
            const int kb4 = jj * TV, rb4 = (rid - jj + 31) * TV;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                fma4(dsv, k4[kb4 + 8 * c + cg], gc[c]);
                fma4(dsv, r4[rb4 + 8 * c + cg], gp[c]);
            }
        }
        // dk, dV of key rid: sums over the 32 query rows
        {
            const int jk = j0 + rid;
            float4 ak[2], av[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) ak[c] = av[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int rr = 0; rr < kQR; ++rr) {
                const float dsv = s_s[rr * kPS + rid], pv = s_p[rr * kPS + rid];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    fma4(dsv, q4u[rr * RV + 8 * c + cg], ak[c]);
                    fma4(pv, d4o[rr * RV + 8 * c + cg], av[c]);
                }
            }
            if (jk < jend) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int t = 32 * c + 4 * cg;
                    if (t < dh) {
                        const float ek[4] = {ak[c].x, ak[c].y, ak[c].z, ak[c].w};
                        const float ev[4] = {av[c].x, av[c].y, av[c].z, av[c].w};
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            if (t + x >= dh) break;
                            if (ek[x] != 0.f) add_at(dk, (bh * K + jk) * dh + t + x, n_kv, 528, scale * ek[x]);
                            if (ev[x] != 0.f) add_at(dv, (bh * K + jk) * dh + t + x, n_kv, 529, ev[x]);
                        }
                    }
                }
            }
        }
        // dR of distance slots rid and rid + 32: pairs (rr, jj = rr - slot + 31)
        for (int sl = rid; sl < kSpan; sl += 32) {
            const long long rrow = (long long)K - 1 - (M + (sl - 31) + i0 - j0);
            if (rrow < 0 || rrow >= K) continue;
            float4 ar[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) ar[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int r_lo = sl > 31 ? sl - 31 : 0, r_hi = sl < 31 ? sl : 31;
            for (int rr = r_lo; rr <= r_hi; ++rr) {
                const float dsv = s_s[rr * kPS + (rr - sl + 31)];
#pragma unroll
                for (int c = 0; c < 2; ++c) fma4(dsv, q4v[rr * RV + 8 * c + cg], ar[c]);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int t = 32 * c + 4 * cg;
                if (t < dh) {
                    const float e[4] = {ar[c].x, ar[c].y, ar[c].z, ar[c].w};
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        if (t + x < dh && e[x] != 0.f) add_at(dr, (rrow * H + h) * dh + t + x, n_r, 530, scale * e[x]);
                }
            }
        }
    }
    {
        const int i = i0 + rid;
        if (i < L) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int t = 32 * c + 4 * cg;
                if (t < dh) {
                    const float ec[4] = {gc[c].x, gc[c].y, gc[c].z, gc[c].w};
                    const float ep[4] = {gp[c].x, gp[c].y, gp[c].z, gp[c].w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        if (t + x >= dh) break;
                        if (TXL_BOUNDS((bh * L + i) * dh + t + x < n_q, 531, (bh * L + i) * dh + t + x))
                            dq[(bh * L + i) * dh + t + x] = scale * (ec[x] + ep[x]);
                        add_at(du, (long long)h * dh + t + x, n_b, 532, scale * ec[x]);
                        add_at(dvb, (long long)h * dh + t + x, n_b, 533, scale * ep[x]);
                    }
                }
            }
        }
    }
}

// Zeroes the summed gradients, then one launch: the block-cooperative kernel
// for d_h <= 64, else one query row per warp.
cudaError_t launch_attn_bwd_simt(const void* q, const void* k, const void* v, const void* r,
                                 const void* ub, const void* vb, const void* dout, int bf16, int B,
                                 int H, int L, int M, int dh, float scale, int lo_shift, float* dq,
                                 float* dk, float* dv, float* dr, float* du, float* dvb,
                                 cudaStream_t stream) {
    const long long K = (long long)M + L;
    const size_t nkv = (size_t)B * H * K * dh * sizeof(float);
    const size_t nr = (size_t)K * H * dh * sizeof(float), nb = (size_t)H * dh * sizeof(float);
    cudaError_t e;
    if ((e = cudaMemsetAsync(dk, 0, nkv, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dv, 0, nkv, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dr, 0, nr, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(du, 0, nb, stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dvb, 0, nb, stream)) != cudaSuccess) return e;
    if (dh <= kDT) {
        static PerDeviceOnce attrs;
        e = attrs.run([] {
            cudaError_t r = cudaFuncSetAttribute(attn_bwd_tiled_kernel<float>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTiledSmem);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(attn_bwd_tiled_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTiledSmem);
            return r;
        });
        if (e != cudaSuccess) return e;
        const long long blocks = (long long)B * H * ((L + kQR - 1) / kQR);
        if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
        if (bf16)
            attn_bwd_tiled_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, kTiledSmem, stream>>>(
                static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(r),
                static_cast<const __nv_bfloat16*>(ub), static_cast<const __nv_bfloat16*>(vb),
                static_cast<const __nv_bfloat16*>(dout), B, H, L, M, dh, scale, lo_shift, dq, dk, dv, dr,
                du, dvb);
        else
            attn_bwd_tiled_kernel<float><<<(unsigned)blocks, 256, kTiledSmem, stream>>>(
                static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
                static_cast<const float*>(r), static_cast<const float*>(ub), static_cast<const float*>(vb),
                static_cast<const float*>(dout), B, H, L, M, dh, scale, lo_shift, dq, dk, dv, dr, du, dvb);
        return cudaGetLastError();
    }
    const long long rows = (long long)B * H * L;
    const long long blocks = (rows + kBwdWarps - 1) / kBwdWarps;
    if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    if (bf16)
        attn_bwd_simt_kernel<__nv_bfloat16><<<(unsigned)blocks, 32 * kBwdWarps, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(r),
            static_cast<const __nv_bfloat16*>(ub), static_cast<const __nv_bfloat16*>(vb),
            static_cast<const __nv_bfloat16*>(dout), B, H, L, M, dh, scale, lo_shift, dq, dk, dv, dr,
            du, dvb);
    else
        attn_bwd_simt_kernel<float><<<(unsigned)blocks, 32 * kBwdWarps, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            static_cast<const float*>(r), static_cast<const float*>(ub), static_cast<const float*>(vb),
            static_cast<const float*>(dout), B, H, L, M, dh, scale, lo_shift, dq, dk, dv, dr, du, dvb);
    return cudaGetLastError();
}

TXL_BOUNDS_READER(bounds_word_attn_bwd)

}  // namespace txl
