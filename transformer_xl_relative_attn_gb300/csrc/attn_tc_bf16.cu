// Fused Transformer-XL relative attention, bf16 in / fp32 accumulate, on the
// sm_103a tensor cores (tcgen05 + TMEM), with TMA-staged K, V and R tiles.
//
// What one CTA computes: one (batch row b, head h, query tile of 128 rows
// i0..i0+127) against all visible keys, swept in key tiles of 64:
//
//   AC(t)    = (q+u) K_t^T                    content terms a + c (64 keys)
//   ring     = (q+v) R_slot^T, one 64-row R slot per key tile
//                                             position terms b + d
//   BD[ii,jj]= band_t[ii, 127 - ii + jj]      the relative shift as an index remap
//   s        = AC + BD (scale * log2 e is folded into q+u and q+v),
//              masked where key j > M + i
//   online softmax over key tiles; O += P V_t on the tensor cores
//
// The score definition follows "Transformer-XL模型 核心源码阅读笔记", section
// "Build the model" (RelPartialLearnableMultiHeadAttn.forward: AC, BD,
// _rel_shift, masked_fill(-inf), softmax, einsum with V) and the
// "Transformer-XL" notes (zty624), sections "Relative Positional Encoding",
// "Relative Shift Trick" and "Causal Mask With Memory".
//
// Position band.  For query row i0+ii and key j0+jj the distance is
// M+i0+ii-j0-jj, i.e. R row (L-i0-128+j0) + (127-ii+jj).  Key tile t (j0 =
// 64t) therefore needs the 191 R rows base+64t .. base+64t+190 (base =
// L-i0-128): three 64-row "slots" g = t, t+1, t+2 of the sequence base+64g.
// Consecutive tiles share two slots, so each tile computes only its newest
// slot (the first tile all three) into a 4-slot ring of TMEM columns: the
// position MMA does exactly the algorithmic work.  Row ii of the band, read
// from band column 127-ii onward, is the shifted position term: the pad /
// reshape / slice of the pages is never performed and no L x (M+L) score
// matrix exists.  R rows outside [0, M+L) are zero-filled by TMA and only land
// on masked entries.
//
// Roles (320 threads, one CTA per SM):
//   warps 0-3  softmax group 0: key tiles 0, 2, 4, ... (one query row per thread)
//   warps 4-7  softmax group 1: key tiles 1, 3, 5, ...
//   warp 8     TMEM allocation; lane 0 issues every MMA
//   warp 9     lane 0 issues the TMA loads into a 3-stage K/V/R ring
// Each group keeps its own running max, sum and O accumulator (TMEM); the two
// partial results are merged at the end.  TMEM columns: AC0 0-63, AC1 64-127,
// position ring 128-383, O0 384-447, O1 448-511.
//
// Every wait is bounded (1 s); on expiry the CTA records a status, drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

namespace tc {
constexpr int BM = 128;        // query rows per CTA (TMEM lanes)
constexpr int BN = 64;         // keys per tile
constexpr int DH = 64;         // head dim: one 128-byte swizzle row
constexpr int SLOT = 64;       // R rows per position slot
constexpr int RING = 4;        // position slots held in TMEM
constexpr int STAGES = 3;
constexpr int NTHREADS = 320;

constexpr uint32_t SZ_Q = BM * DH * 2;      // 16 KB
constexpr uint32_t SZ_T = BN * DH * 2;      //  8 KB: one K, V or R slot tile
constexpr uint32_t SZ_STAGE = 3 * SZ_T;     // K, V, R slot
constexpr uint32_t SZ_P = BM * BN * 2;      // 16 KB per group
constexpr uint32_t OFF_QU = 0;
constexpr uint32_t OFF_QV = OFF_QU + SZ_Q;
constexpr uint32_t OFF_STAGE = OFF_QV + SZ_Q;
constexpr uint32_t OFF_PRO = OFF_STAGE + STAGES * SZ_STAGE;  // R slots 0, 1 of the first tile
constexpr uint32_t OFF_P = OFF_PRO + 2 * SZ_T;
constexpr uint32_t OFF_BAR = OFF_P + 2 * SZ_P;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;

constexpr uint32_t COL_AC = 0;      // + 64 * group
constexpr uint32_t COL_RING = 128;  // + 64 * slot
constexpr uint32_t COL_O = 384;     // + 64 * group
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t IDESC_N64 = idesc_bf16_f32(128, 64, 0);  // K-major B (K, R)
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, DH, 1);   // MN-major B (V)

constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales
}  // namespace tc

struct TcParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* ub;
    const __nv_bfloat16* vb;
    __nv_bfloat16* out;
    int B, H, L, M;
    int n_qtiles;
    float scale_log2;  // scale * log2(e), folded into q+u and q+v
    int inject;        // 1: withhold the first score-ready signal (timeout test)
    int* status;       // device status word
};

struct TcShared {
    uint64_t full[tc::STAGES];
    uint64_t empty[tc::STAGES];
    uint64_t q_ready;
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Bounded wait that ignores the abort flag: used to drain in-flight copies and
// MMAs before the CTA releases its shared and tensor memory.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            record_status(status, kDevTimeoutDrain);
            return;
        }
    }
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a.x + b.x, a.y + b.y) in one packed instruction
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}

__global__ void __launch_bounds__(tc::NTHREADS, 1)
attn_tc_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmR, const TcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    TcShared* sh = reinterpret_cast<TcShared*>(smem + OFF_BAR);
    const uint32_t s_base = smem_u32(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // Work item: longest query tiles first (they see the most keys).
    const int n_bh = p.B * p.H;
    const int item = blockIdx.x;
    const int qt = p.n_qtiles - 1 - item / n_bh;
    const int bh = item % n_bh;
    const int h = bh % p.H;
    const int i0 = qt * BM;
    const int rows_valid = min(BM, p.L - i0);
    const int kmax = p.M + i0 + rows_valid - 1;  // last key any row of the tile sees
    const int ntiles = kmax / BN + 1;
    const int rbase = p.L - i0 - BM;             // R row of slot 0, position 0

    if (warp == 8) {
        tmem_alloc(&sh->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], 1);
        }
        mbar_init(&sh->q_ready, 2 * BM);
        for (int g = 0; g < 2; ++g) {
            mbar_init(&sh->s_full[g], 1);
            mbar_init(&sh->p_full[g], BM);
        }
        mbar_init(&sh->o_done, 1);
        mbar_init(&sh->drain, 1);
        sh->abort = 0;
        fence_mbar_init();
    }
    if (warp == 9 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmR);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;

    if (warp < 8) {
        // ------------------------------------------------------ softmax groups
        const int grp = warp >> 2;          // 0: even key tiles, 1: odd key tiles
        const int wq = warp & 3;            // TMEM lane quarter
        const int ii = tid & 127;           // query row within the tile
        const int i = i0 + ii;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        // Group 0 writes (q+u)*c, group 1 (q+v)*c (c = scale*log2 e), rounded
        // to bf16, as 128-byte swizzled rows (chunk c of row ii at c ^ (ii&7)).
        {
            const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((size_t)bh * p.L + i) * DH);
            const uint4* brow =
                reinterpret_cast<const uint4*>((grp == 0 ? p.ub : p.vb) + (size_t)h * DH);
            const uint32_t dst = s_base + (grp == 0 ? OFF_QU : OFF_QV) + ii * 128;
            const float c = p.scale_log2;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 q4 = make_uint4(0, 0, 0, 0);
                if (i < p.L) q4 = qrow[ch];
                const uint4 b4 = brow[ch];
                const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&q4);
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b4);
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 qf = __bfloat1622float2(q2[e]);
                    const float2 bf = __bfloat1622float2(b2[e]);
                    w[e] = pack_bf16x2((qf.x + bf.x) * c, (qf.y + bf.y) * c);
                }
                st_shared_v4(dst + ((ch ^ (ii & 7)) << 4), w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&sh->q_ready);
        }

        float m_run = -INFINITY;  // running max (log2 domain), may lag the true max by < 8
        float l_run = 0.f;
        bool ok = true;
        int it = 0;
        const uint32_t p_tile = s_base + OFF_P + grp * SZ_P;
        for (int t = grp; t < ntiles; t += 2, ++it) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&sh->s_full[grp], it & 1, kDevTimeoutSoftmax, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            const int j0 = t * BN;
            const bool need_mask = (j0 + BN - 1) > (p.M + i0);
            const int jlim = p.M + i - j0;  // keys jj > jlim are masked
            float sc[BN];
            float tmax = -INFINITY;
#pragma unroll
            for (int q2 = 0; q2 < BN / 32; ++q2) {
                uint32_t ac[32], w0[32], w1[32];
                tmem_ld32(tmem + lane_off + COL_AC + 64 * grp + 32 * q2, ac);
                // band columns c0 .. c0+63 of this tile, c0 = 96 - 32*wq + 32*q2
                const int cA = 96 - 32 * wq + 32 * q2, cB = cA + 32;
                const uint32_t rA = COL_RING + 64 * ((t + (cA >> 6)) & (RING - 1)) + (cA & 63);
                const uint32_t rB = COL_RING + 64 * ((t + (cB >> 6)) & (RING - 1)) + (cB & 63);
                tmem_ld32(tmem + lane_off + rA, w0);
                tmem_ld32(tmem + lane_off + rB, w1);
                tmem_wait_ld();
                float win[64];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    win[x] = __uint_as_float(w0[x]);
                    win[32 + x] = __uint_as_float(w1[x]);
                }
                // per-row shift by o = 31 - lane: win[x] <- win[x + o]
                const int o = 31 - lane;
#pragma unroll
                for (int sb = 16; sb >= 1; sb >>= 1) {
                    const bool take = (o & sb) != 0;
#pragma unroll
                    for (int x = 0; x < 32 + sb - 1; ++x) win[x] = take ? win[x + sb] : win[x];
                }
#pragma unroll
                for (int x = 0; x < 32; x += 2) {
                    const float2 s2 = add2(make_float2(__uint_as_float(ac[x]), __uint_as_float(ac[x + 1])),
                                           make_float2(win[x], win[x + 1]));
                    sc[32 * q2 + x] = s2.x;
                    sc[32 * q2 + x + 1] = s2.y;
                }
                if (need_mask) {
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (32 * q2 + x > jlim) sc[32 * q2 + x] = -INFINITY;
                }
#pragma unroll
                for (int x = 0; x < 32; x += 2) tmax = max3(tmax, sc[32 * q2 + x], sc[32 * q2 + x + 1]);
            }
            // Conditional rescale: keep the running max unless the tile's max
            // exceeds it by more than the threshold (then p <= 2^threshold).
            const float m_new = (tmax > m_run + kRescaleThreshold) ? tmax : m_run;
            // A row may have seen no visible key yet in this group (m_new = -inf):
            // exponentiate against 0 instead, so every p is exactly 0, not NaN.
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_run - m_use);  // 0 until the first visible key, else 1 or < 1
            if (it > 0 && __any_sync(0xffffffffu, m_new != m_run)) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o32[32];
                    tmem_ld32(tmem + lane_off + COL_O + 64 * grp + 32 * c, o32);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        o32[x] = __float_as_uint(__uint_as_float(o32[x]) * alpha);
                    tmem_st32(tmem + lane_off + COL_O + 64 * grp + 32 * c, o32);
                }
                tmem_wait_st();
            }
            const float2 negm = make_float2(-m_use, -m_use);
            float2 rs = make_float2(0.f, 0.f);
#pragma unroll
            for (int c8 = 0; c8 < BN / 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = add2(make_float2(sc[c8 * 8 + 2 * e], sc[c8 * 8 + 2 * e + 1]), negm);
                    const float p0 = ex2(x.x), p1 = ex2(x.y);
                    rs = add2(rs, make_float2(p0, p1));
                    w[e] = pack_bf16x2(p0, p1);
                }
                st_shared_v4(p_tile + ii * 128 + ((c8 ^ (ii & 7)) << 4), w[0], w[1], w[2], w[3]);
            }
            l_run = l_run * alpha + (rs.x + rs.y);
            m_run = m_new;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sh->p_full[grp]);
        }
        // ------------------------------------------------------ merge + store
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&sh->o_done, 0, kDevTimeoutSoftmax, abort, p.status));
        // the two groups exchange (m, l, O) through the (now idle) stage buffers
        float* xch = reinterpret_cast<float*>(smem + OFF_STAGE);  // [128][66] floats
        if (ok) {
            tc_fence_after();
            uint32_t o0[32], o1[32];
            const bool had = grp < ntiles;  // group 1 has no tile when ntiles == 1
            tmem_ld32(tmem + lane_off + COL_O + 64 * grp, o0);
            tmem_ld32(tmem + lane_off + COL_O + 64 * grp + 32, o1);
            tmem_wait_ld();
            if (grp == 1) {
                float* row = xch + ii * 66;
                row[0] = had ? m_run : -INFINITY;
                row[1] = had ? l_run : 0.f;
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    row[2 + x] = had ? __uint_as_float(o0[x]) : 0.f;
                    row[34 + x] = had ? __uint_as_float(o1[x]) : 0.f;
                }
            }
        }
        // both groups reach this barrier on every path (ok is warp-uniform)
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (ok && grp == 0) {
            uint32_t o0[32], o1[32];
            tmem_ld32(tmem + lane_off + COL_O, o0);
            tmem_ld32(tmem + lane_off + COL_O + 32, o1);
            tmem_wait_ld();
            const float* row = xch + ii * 66;
            const float m1 = row[0], l1 = row[1];
            const float m = fmaxf(m_run, m1);
            const float f0 = ex2(m_run - m), f1 = ex2(m1 - m);
            const float inv = 1.f / (l_run * f0 + l1 * f1);
            const float a0 = f0 * inv, a1 = f1 * inv;
            if (i < p.L) {
                uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)bh * p.L + i) * DH);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int x = 8 * c + e;
                        const float mine = __uint_as_float(x < 32 ? o0[x] : o1[x - 32]);
                        v[e] = mine * a0 + row[2 + x] * a1;
                    }
                    uint4 w;
                    w.x = pack_bf16x2(v[0], v[1]);
                    w.y = pack_bf16x2(v[2], v[3]);
                    w.z = pack_bf16x2(v[4], v[5]);
                    w.w = pack_bf16x2(v[6], v[7]);
                    orow[c] = w;
                }
            }
        }
        tc_fence_before();
    } else if (warp == 8) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a_qu = s_base + OFF_QU, a_qv = s_base + OFF_QV;
            bool ok = mbar_wait(&sh->q_ready, 0, kDevTimeoutMma, abort, p.status);
            tc_fence_after();
            // S(t): content MMA into AC[t&1], newest position slot(s) into the ring
            auto issue_s = [&](int t) -> bool {
                const int s = t % STAGES;
                if (!mbar_wait(&sh->full[s], (t / STAGES) & 1, kDevTimeoutMma, abort, p.status))
                    return false;
                tc_fence_after();
                const uint32_t sK = s_base + OFF_STAGE + s * SZ_STAGE;
                const uint32_t sR = sK + 2 * SZ_T;
#pragma unroll
                for (int k = 0; k < DH / 16; ++k)
                    mma_bf16(tmem + COL_AC + 64 * (t & 1), smem_desc_sw128(a_qu + 32 * k, 16, 1024),
                             smem_desc_sw128(sK + 32 * k, 16, 1024), IDESC_N64, k > 0);
                if (t == 0) {
                    for (int g = 0; g < 2; ++g) {
                        const uint32_t sRp = s_base + OFF_PRO + g * SZ_T;
#pragma unroll
                        for (int k = 0; k < DH / 16; ++k)
                            mma_bf16(tmem + COL_RING + 64 * g, smem_desc_sw128(a_qv + 32 * k, 16, 1024),
                                     smem_desc_sw128(sRp + 32 * k, 16, 1024), IDESC_N64, k > 0);
                    }
                }
                const int gslot = t + 2;
#pragma unroll
                for (int k = 0; k < DH / 16; ++k)
                    mma_bf16(tmem + COL_RING + 64 * (gslot & (RING - 1)),
                             smem_desc_sw128(a_qv + 32 * k, 16, 1024),
                             smem_desc_sw128(sR + 32 * k, 16, 1024), IDESC_N64, k > 0);
                if (!(p.inject == 1 && t == 0)) mma_commit(&sh->s_full[t & 1]);
                return true;
            };
            for (int t = 0; ok && t < 2 && t < ntiles; ++t) ok = issue_s(t);
            for (int t = 0; ok && t < ntiles; ++t) {
                const int g = t & 1;
                if (!mbar_wait(&sh->p_full[g], (t >> 1) & 1, kDevTimeoutMma, abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int s = t % STAGES;
                const uint32_t sV = s_base + OFF_STAGE + s * SZ_STAGE + SZ_T;
                const uint32_t aP = s_base + OFF_P + g * SZ_P;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_bf16(tmem + COL_O + 64 * g, smem_desc_sw128(aP + 32 * k, 16, 1024),
                             smem_desc_sw128(sV + k * 2048, BN * 128, 1024), IDESC_PV,
                             (t > 1 || k > 0) ? 1u : 0u);
                mma_commit(&sh->empty[s]);
                if (t + 2 < ntiles) ok = issue_s(t + 2);
            }
            if (ok) mma_commit(&sh->o_done);
            mma_commit(&sh->drain);
            drain_wait(&sh->drain, 0, p.status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % STAGES;
                if (t >= STAGES && !mbar_wait(&sh->empty[s], ((t / STAGES) & 1) ^ 1,
                                              kDevTimeoutProducer, abort, p.status))
                    break;
                uint8_t* st = smem + OFF_STAGE + s * SZ_STAGE;
                mbar_expect_tx(&sh->full[s], SZ_STAGE + (t == 0 ? 2 * SZ_T : 0));
                const int j0 = t * BN;
                tma_load_3d(st, &tmK, &sh->full[s], 0, j0, bh);
                tma_load_3d(st + SZ_T, &tmV, &sh->full[s], 0, j0, bh);
                tma_load_2d(st + 2 * SZ_T, &tmR, &sh->full[s], h * DH, rbase + SLOT * (t + 2));
                if (t == 0) {
                    tma_load_2d(smem + OFF_PRO, &tmR, &sh->full[s], h * DH, rbase);
                    tma_load_2d(smem + OFF_PRO + SZ_T, &tmR, &sh->full[s], h * DH, rbase + SLOT);
                }
                issued = t + 1;
            }
            // drain: the last load of each stage has landed
            for (int t = issued - STAGES; t < issued; ++t)
                if (t >= 0) drain_wait(&sh->full[t % STAGES], (t / STAGES) & 1, p.status);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

static bool encode_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                        const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                    strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Returns cudaErrorInvalidValue if a tensor map cannot be encoded.
cudaError_t launch_attn_tc_bf16(const void* q, const void* k, const void* v, const void* r,
                                const void* ub, const void* vb, int B, int H, int L, int M,
                                float scale, void* out, int inject, int* status,
                                cudaStream_t stream) {
    using namespace tc;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_bf16_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int K = M + L;
    CUtensorMap mK, mV, mR;
    {
        cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)K, (cuuint64_t)B * H};
        cuuint64_t strides[2] = {(cuuint64_t)DH * 2, (cuuint64_t)K * DH * 2};
        cuuint32_t box[3] = {DH, BN, 1};
        if (!encode_bf16(&mK, k, 3, dims, strides, box)) return cudaErrorInvalidValue;
        if (!encode_bf16(&mV, v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)H * DH, (cuuint64_t)K};
        cuuint64_t strides[1] = {(cuuint64_t)H * DH * 2};
        cuuint32_t box[2] = {DH, SLOT};
        if (!encode_bf16(&mR, r, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    TcParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.ub = static_cast<const __nv_bfloat16*>(ub);
    p.vb = static_cast<const __nv_bfloat16*>(vb);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.B = B;
    p.H = H;
    p.L = L;
    p.M = M;
    p.n_qtiles = (L + BM - 1) / BM;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.inject = inject;
    p.status = status;
    const long long grid = (long long)B * H * p.n_qtiles;
    if (grid > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    attn_tc_bf16_kernel<<<(unsigned)grid, NTHREADS, SMEM_BYTES, stream>>>(mK, mV, mR, p);
    return cudaGetLastError();
}

}  // namespace txl
