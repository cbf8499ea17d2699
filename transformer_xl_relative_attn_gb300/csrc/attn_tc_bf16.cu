// Fused Transformer-XL relative attention, bf16 in / fp32 accumulate, on the
// sm_103a tensor cores (tcgen05 + TMEM), with TMA-staged K, V and R tiles.
//
// What one CTA computes: one (batch row b, head h, query tile of 128 rows
// i0..i0+127) against all visible keys, swept in key tiles of 128:
//
//   AC   = (q+u) K_tile^T                 content terms a + c
//   Band = (q+v) R_band^T                 position terms b + d, for the 255
//                                         distances this tile can meet
//   BD[ii, jj] = Band[ii, 127 - ii + jj]  the relative shift as an index remap
//   s    = scale (AC + BD), masked where key j > M + i
//   online softmax over key tiles; O += P V_tile on the tensor cores
//
// The score definition follows "Transformer-XL模型 核心源码阅读笔记", section
// "Build the model" (RelPartialLearnableMultiHeadAttn.forward: AC, BD,
// _rel_shift, masked_fill(-inf), softmax, einsum with V) and the "Transformer-XL"
// notes (zty624), sections "Relative Positional Encoding", "Relative Shift
// Trick" and "Causal Mask With Memory".
//
// Why the band: for query row i0+ii and key j0+jj the distance is
// M+i0+ii-j0-jj, i.e. R row (L-i0+j0-128) + (127-ii+jj).  Loading the 256 R
// rows from r_lo = L-i0+j0-128 gives one dense MMA whose row ii, read from
// column 127-ii onward, is exactly the shifted position term.  The pad /
// reshape / slice of the pages is never performed and no L x (M+L) score
// matrix exists.  R rows outside [0, M+L) (negative distances or past the
// table) are zero-filled by TMA and only ever land on masked entries.
//
// Roles (192 threads): warps 0-3 own one query row per thread (TMEM lane =
// row) and do the remap, mask, softmax, O rescale and epilogue; warp 4
// allocates TMEM and one lane issues every MMA; one lane of warp 5 issues the
// TMA loads into a 2-stage K/V/R ring.  Every wait is bounded (1 s); on expiry
// the CTA records a status, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

namespace tc {
constexpr int BM = 128;          // query rows per tile (TMEM lanes)
constexpr int BN = 128;          // keys per tile
constexpr int DH = 64;           // head dim: one 128-byte swizzle row
constexpr int BAND = BM + BN;    // R rows loaded per key tile (255 used)
constexpr int STAGES = 2;

constexpr uint32_t SZ_Q = BM * DH * 2;
constexpr uint32_t SZ_K = BN * DH * 2;
constexpr uint32_t SZ_V = BN * DH * 2;
constexpr uint32_t SZ_R = BAND * DH * 2;
constexpr uint32_t SZ_STAGE = SZ_K + SZ_V + SZ_R;
constexpr uint32_t SZ_PHALF = BM * 64 * 2;  // 64 keys of P per swizzle-row block
constexpr uint32_t OFF_QU = 0;
constexpr uint32_t OFF_QV = OFF_QU + SZ_Q;
constexpr uint32_t OFF_STAGE = OFF_QV + SZ_Q;
constexpr uint32_t OFF_P = OFF_STAGE + STAGES * SZ_STAGE;
constexpr uint32_t OFF_BAR = OFF_P + 2 * SZ_PHALF;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;  // + barriers + alignment slack

constexpr uint32_t COL_AC = 0;
constexpr uint32_t COL_BAND = 128;
constexpr uint32_t COL_O = 384;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t IDESC_AC = idesc_bf16_f32(128, BN, 0);
constexpr uint32_t IDESC_BAND = idesc_bf16_f32(128, BAND, 0);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, DH, 1);
}  // namespace tc

struct TcParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* ub;
    const __nv_bfloat16* vb;
    __nv_bfloat16* out;
    int B, H, L, M;
    int n_qtiles;
    float scale_log2;  // scale * log2(e)
    int inject;        // 1: withhold the first score-ready signal (timeout test)
    int* status;       // device status word
};

struct TcShared {
    uint64_t full[tc::STAGES];
    uint64_t empty[tc::STAGES];
    uint64_t q_ready;
    uint64_t s_full;
    uint64_t p_full;
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

__global__ void __launch_bounds__(192, 1)
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

    if (warp == 4) {
        tmem_alloc(&sh->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], 1);
        }
        mbar_init(&sh->q_ready, BM);
        mbar_init(&sh->s_full, 1);
        mbar_init(&sh->p_full, BM);
        mbar_init(&sh->o_done, 1);
        mbar_init(&sh->drain, 1);
        sh->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmR);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;

    if (warp < 4) {
        // ------------------------------------------------------ softmax rows
        const int ii = tid;
        const int i = i0 + ii;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        // Qu = q + u and Qv = q + v, rounded to bf16, written as 128-byte
        // swizzled rows (16-byte chunk c of row ii at chunk c ^ (ii & 7)).
        {
            const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((size_t)bh * p.L + i) * DH);
            const uint4* urow = reinterpret_cast<const uint4*>(p.ub + (size_t)h * DH);
            const uint4* vrow = reinterpret_cast<const uint4*>(p.vb + (size_t)h * DH);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 qv4 = make_uint4(0, 0, 0, 0);
                if (i < p.L) qv4 = qrow[c];
                const uint4 u4 = urow[c], v4 = vrow[c];
                const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qv4);
                const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&u4);
                const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&v4);
                uint32_t wu[4], wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 qf = __bfloat1622float2(q2[e]);
                    const float2 uf = __bfloat1622float2(u2[e]);
                    const float2 vf = __bfloat1622float2(v2[e]);
                    wu[e] = pack_bf16x2(qf.x + uf.x, qf.y + uf.y);
                    wv[e] = pack_bf16x2(qf.x + vf.x, qf.y + vf.y);
                }
                const uint32_t off = ii * 128 + ((c ^ (ii & 7)) << 4);
                st_shared_v4(s_base + OFF_QU + off, wu[0], wu[1], wu[2], wu[3]);
                st_shared_v4(s_base + OFF_QV + off, wv[0], wv[1], wv[2], wv[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&sh->q_ready);
        }

        float m_run = -INFINITY;  // running max, log2 domain
        float l_run = 0.f;        // running sum of probabilities
        bool ok = true;
        for (int t = 0; t < ntiles && ok; ++t) {
            // the warp continues only if every lane saw the signal: the
            // tcgen05.ld below is warp-collective
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&sh->s_full, t & 1, kDevTimeoutSoftmax, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            const int j0 = t * BN;
            const bool need_mask = (j0 + BN - 1) > (p.M + i0);
            const int jlim = p.M + i - j0;  // keys jj > jlim are masked
            float sc[BN];
            float tmax = -INFINITY;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t ac[32], w0[32], w1[32];
                tmem_ld32(tmem + lane_off + COL_AC + 32 * q4, ac);
                const uint32_t wcol = COL_BAND + 96 - 32 * warp + 32 * q4;
                tmem_ld32(tmem + lane_off + wcol, w0);
                tmem_ld32(tmem + lane_off + wcol + 32, w1);
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
                for (int x = 0; x < 32; ++x) {
                    float s = (__uint_as_float(ac[x]) + win[x]) * p.scale_log2;
                    if (need_mask && (32 * q4 + x) > jlim) s = -INFINITY;
                    sc[32 * q4 + x] = s;
                    tmax = fmaxf(tmax, s);
                }
            }
            const float m_new = fmaxf(m_run, tmax);
            const float alpha = exp2f(m_run - m_new);
            // Rescale the running output when the max grew (warp-collective).
            if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o32[32];
                    tmem_ld32(tmem + lane_off + COL_O + 32 * c, o32);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        o32[x] = __float_as_uint(__uint_as_float(o32[x]) * alpha);
                    tmem_st32(tmem + lane_off + COL_O + 32 * c, o32);
                }
                tmem_wait_st();
            }
            float rsum = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < BN / 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = exp2f(sc[c8 * 8 + 2 * e] - m_new);
                    const float p1 = exp2f(sc[c8 * 8 + 2 * e + 1] - m_new);
                    rsum += p0 + p1;
                    w[e] = pack_bf16x2(p0, p1);
                }
                const uint32_t half = c8 >> 3, ch = c8 & 7;
                const uint32_t addr = s_base + OFF_P + half * SZ_PHALF + ii * 128 + ((ch ^ (ii & 7)) << 4);
                st_shared_v4(addr, w[0], w[1], w[2], w[3]);
            }
            l_run = l_run * alpha + rsum;
            m_run = m_new;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sh->p_full);
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&sh->o_done, 0, kDevTimeoutSoftmax, abort, p.status));
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l_run;
            uint32_t o0[32], o1[32];
            tmem_ld32(tmem + lane_off + COL_O, o0);
            tmem_ld32(tmem + lane_off + COL_O + 32, o1);
            tmem_wait_ld();
            if (i < p.L) {
                uint4* orow = reinterpret_cast<uint4*>(p.out + ((size_t)bh * p.L + i) * DH);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t* src = (c < 4) ? &o0[8 * c] : &o1[8 * (c - 4)];
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
                    orow[c] = w;
                }
            }
        }
        tc_fence_before();
    } else if (warp == 4) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(&sh->q_ready, 0, kDevTimeoutMma, abort, p.status);
            tc_fence_after();
            const uint32_t a_qu = s_base + OFF_QU, a_qv = s_base + OFF_QV;
            int t = 0;
            for (; ok && t < ntiles; ++t) {
                const int s = t & 1;
                if (!mbar_wait(&sh->full[s], (t >> 1) & 1, kDevTimeoutMma, abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sK = s_base + OFF_STAGE + s * SZ_STAGE;
                const uint32_t sV = sK + SZ_K;
                const uint32_t sR = sV + SZ_V;
#pragma unroll
                for (int k = 0; k < DH / 16; ++k)
                    mma_bf16(tmem + COL_AC, smem_desc_sw128(a_qu + 32 * k, 16, 1024),
                             smem_desc_sw128(sK + 32 * k, 16, 1024), IDESC_AC, k > 0);
#pragma unroll
                for (int k = 0; k < DH / 16; ++k)
                    mma_bf16(tmem + COL_BAND, smem_desc_sw128(a_qv + 32 * k, 16, 1024),
                             smem_desc_sw128(sR + 32 * k, 16, 1024), IDESC_BAND, k > 0);
                if (!(p.inject == 1 && t == 0)) mma_commit(&sh->s_full);
                if (!mbar_wait(&sh->p_full, t & 1, kDevTimeoutMma, abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t aP = s_base + OFF_P;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_bf16(tmem + COL_O,
                             smem_desc_sw128(aP + (k >> 2) * SZ_PHALF + (k & 3) * 32, 16, 1024),
                             smem_desc_sw128(sV + k * 2048, BN * 128, 1024), IDESC_PV,
                             (t > 0 || k > 0) ? 1u : 0u);
                mma_commit(&sh->empty[s]);
            }
            if (ok) mma_commit(&sh->o_done);
            // drain: every MMA issued above has completed before TMEM is freed
            mma_commit(&sh->drain);
            drain_wait(&sh->drain, 0, p.status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t & 1;
                if (t >= STAGES &&
                    !mbar_wait(&sh->empty[s], ((t >> 1) & 1) ^ 1, kDevTimeoutProducer, abort, p.status))
                    break;
                uint8_t* st = smem + OFF_STAGE + s * SZ_STAGE;
                mbar_expect_tx(&sh->full[s], SZ_STAGE);
                const int j0 = t * BN;
                tma_load_3d(st, &tmK, &sh->full[s], 0, j0, bh);
                tma_load_3d(st + SZ_K, &tmV, &sh->full[s], 0, j0, bh);
                tma_load_2d(st + SZ_K + SZ_V, &tmR, &sh->full[s], h * DH, p.L - i0 + j0 - BM);
                issued = t + 1;
            }
            // drain: the last load of each stage has landed
            for (int t = issued - STAGES; t < issued; ++t)
                if (t >= 0) drain_wait(&sh->full[t & 1], (t >> 1) & 1, p.status);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
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
        cuuint32_t box[2] = {DH, BAND};
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
    attn_tc_bf16_kernel<<<(unsigned)grid, 192, SMEM_BYTES, stream>>>(mK, mV, mR, p);
    return cudaGetLastError();
}

}  // namespace txl
