// Projections that feed the relative attention, on the sm_103a tensor cores:
//
//   q = h W_q^T                     -> [B, H, L, d_h]
//   k = [mem; h] W_k^T, v likewise  -> [B, H, M+L, d_h], memory rows first
//   r = emb W_r^T                   -> [M+L, H, d_h]
//
// ("Transformer-XL模型 核心源码阅读笔记", RelPartialLearnableMultiHeadAttn.forward:
// qkv_net over the concatenation of memory and current hidden states, r_net over
// the position embedding; "Transformer-XL" notes, section "Batched Tensor
// Contract".)  The memory rows and the current rows are two row sources of one
// GEMM, so no [mem; h] concatenation is formed, and the epilogue writes each
// 64-column head slice straight into the head-split layout.
//
// One CTA per SM walks output tiles of 128 rows x 256 columns; K (= d) is
// streamed in 64-element steps through a 4-stage TMA ring (A tile 16 KB, B tile
// 32 KB, 128B swizzle).  Roles (256 threads): warp 0 lane 0 issues the TMA
// loads, warp 1 issues the MMAs (whole warp, one elected lane: M=128, N=256,
// K=16 per instruction into a TMEM accumulator), warps 4-7 drain the
// accumulator (one row per thread) to bf16 global stores.  Two accumulators of
// 256 columns let the epilogue of one tile overlap the MMAs of the next.
// Every wait is bounded (1 s) and reports through the device status word.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

namespace pg {
constexpr int BM = 128;     // rows per tile (TMEM lanes)
constexpr int BN = 256;     // columns per tile (MMA N)
constexpr int BK = 64;      // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int NTHREADS = 256;
constexpr uint32_t SZ_A = BM * BK * 2;  // 16 KB
constexpr uint32_t SZ_B = BN * BK * 2;  // 32 KB
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * SZ_A;
constexpr uint32_t OFF_BAR = OFF_B + STAGES * SZ_B;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one sm_103a CTA");
constexpr uint32_t TMEM_COLS = 512;     // two accumulators of BN columns
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, 0);
}  // namespace pg

struct PgParams {
    int B;          // batch rows
    int Ta, Tb;     // rows per batch from source a (memory) then source b (current)
    int K;          // reduction length (= d)
    int N;          // output columns (a multiple of BN)
    int d, H, dh;   // output column c -> tensor c / d, head (c % d) / dh, element c % dh
    int T_out;      // rows per (batch, head) of the outputs
    int plain;      // 1: outputs are [rows, d] row-major (no head split)
    int n_rt, n_nt, n_tiles;
    __nv_bfloat16* out[3];
    int* status;
};

struct PgShared {
    uint64_t full[pg::STAGES];
    uint64_t empty[pg::STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Tile w of the launch: column tile fastest, then row tile, then batch row.
__device__ __forceinline__ void pg_tile(const PgParams& p, int w, int& b, int& t0, int& n0) {
    const int nt = w % p.n_nt, rest = w / p.n_nt;
    n0 = nt * pg::BN;
    t0 = (rest % p.n_rt) * pg::BM;
    b = rest / p.n_rt;
}

__global__ void __launch_bounds__(pg::NTHREADS, 1)
proj_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAb,
                 const __grid_constant__ CUtensorMap tmW, const PgParams p) {
    using namespace pg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    PgShared* sh = reinterpret_cast<PgShared*>(smem + OFF_BAR);
    const uint32_t s_base = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ksteps = p.K / BK;

    if (warp == 1) {
        tmem_alloc(&sh->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh->acc_full[a], 1);
            mbar_init(&sh->acc_empty[a], 4);  // one arrival per epilogue warp
        }
        mbar_init(&sh->drain, 1);
        sh->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmAb);
        tma_prefetch_desc(&tmW);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            bool ok = true;
            int c = 0;  // loads issued into the ring
            for (int w = blockIdx.x; ok && w < p.n_tiles; w += gridDim.x) {
                int b, t0, n0;
                pg_tile(p, w, b, t0, n0);
                // a row tile lies wholly in one source (Ta is a multiple of BM)
                const bool from_a = t0 < p.Ta;
                for (int k = 0; k < ksteps; ++k, ++c) {
                    const int s = c % STAGES;
                    if (c >= STAGES && !mbar_wait(&sh->empty[s], ((c / STAGES) & 1) ^ 1,
                                                  kDevTimeoutProducer, abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&sh->full[s], SZ_A + SZ_B);
                    if (from_a)
                        tma_load_3d(smem + OFF_A + s * SZ_A, &tmA, &sh->full[s], k * BK, t0, b);
                    else
                        tma_load_3d(smem + OFF_A + s * SZ_A, &tmAb, &sh->full[s], k * BK, t0 - p.Ta, b);
                    tma_load_2d(smem + OFF_B + s * SZ_B, &tmW, &sh->full[s], k * BK, n0);
                }
            }
            // drain: the last load into each ring slot has landed
            for (int i = c - STAGES; i < c; ++i)
                if (i >= 0) {
                    const uint64_t t0n = globaltimer_ns();
                    while (!mbar_try_wait(&sh->full[i % STAGES], (i / STAGES) & 1))
                        if (globaltimer_ns() - t0n > kWaitLimitNs) {
                            record_status(p.status, kDevTimeoutDrain);
                            break;
                        }
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        const uint32_t leader = elect_one();
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok)
                ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kDevTimeoutMma, abort, p.status));
            return ok;
        };
        const uint64_t dA0 = smem_desc_sw128(s_base + OFF_A, 16, 1024);
        const uint64_t dB0 = smem_desc_sw128(s_base + OFF_B, 16, 1024);
        int c = 0, j = 0;  // k-steps consumed; tiles done by this CTA
        for (int w = blockIdx.x; ok && w < p.n_tiles; w += gridDim.x, ++j) {
            const int acc = j & 1;
            // the epilogue has drained this accumulator's previous tile
            if (j >= 2 && !wait(&sh->acc_empty[acc], ((j >> 1) - 1) & 1)) break;
            tc_fence_after();
            const uint32_t d_acc = tmem + acc * BN;
            for (int k = 0; k < ksteps; ++k, ++c) {
                const int s = c % STAGES;
                if (!wait(&sh->full[s], (c / STAGES) & 1)) break;
                tc_fence_after();
                const uint64_t a = dA0 + s * (SZ_A >> 4), bdesc = dB0 + s * (SZ_B >> 4);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_ss_elect(d_acc, a + 2 * kk, bdesc + 2 * kk, IDESC, (k > 0 || kk > 0) ? 1u : 0u,
                                 leader);
                if (leader) mma_commit(&sh->empty[s]);
            }
            if (!ok) break;
            if (leader) mma_commit(&sh->acc_full[acc]);
        }
        if (leader) mma_commit(&sh->drain);
        const uint64_t t0n = globaltimer_ns();
        while (!mbar_try_wait(&sh->drain, 0))
            if (globaltimer_ns() - t0n > kWaitLimitNs) {
                record_status(p.status, kDevTimeoutDrain);
                break;
            }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------- epilogue
        const int wq = warp & 3;
        const int row = wq * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        bool ok = true;
        int j = 0;
        for (int w = blockIdx.x; ok && w < p.n_tiles; w += gridDim.x, ++j) {
            const int acc = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&sh->acc_full[acc], (j >> 1) & 1,
                                                   kDevTimeoutSoftmax, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            int b, t0, n0;
            pg_tile(p, w, b, t0, n0);
            const int t = t0 + row;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + acc * BN + 32 * cc, v);
                tmem_wait_ld();
                if (cc == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
                }
                const int n = n0 + 32 * cc;
                const int o = n / p.d, nd = n - o * p.d;
                __nv_bfloat16* const base = o == 0 ? p.out[0] : (o == 1 ? p.out[1] : p.out[2]);
                __nv_bfloat16* dst;
                if (p.plain) {
                    dst = base + ((size_t)b * p.T_out + t) * p.d + nd;
                } else {
                    const int head = nd / p.dh, e = nd - head * p.dh;
                    dst = base + (((size_t)b * p.H + head) * p.T_out + t) * p.dh + e;
                }
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 w4;
                    w4.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
                    w4.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
                    w4.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
                    w4.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
                    d4[q] = w4;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*PgEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                               CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                               CUtensorMapFloatOOBfill);

static PgEncodeFn pg_encode_fn() {
    static PgEncodeFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PgEncodeFn>(ptr);
    }
    return fn;
}

static bool pg_encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box) {
    PgEncodeFn fn = pg_encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int pg_num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
    }
    return n;
}

// out[c / d] <- rows of [a_src; b_src] (per batch row: Ta rows of a_src, then Tb
// rows of b_src, each row K bf16) times w^T (w: N rows of K, row-major).
// Requires Ta, Tb multiples of 128 (Ta may be 0), K a multiple of 64, N a
// multiple of 256, N / d <= 3.
cudaError_t launch_proj_gemm(const void* a_src, int Ta, const void* b_src, int Tb, int B,
                             const void* w, int N, int K, int d, int H, int dh, int T_out, int plain,
                             void* out0, void* out1, void* out2, int* status, cudaStream_t stream) {
    using namespace pg;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(proj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap mA, mB, mW;
    const cuuint32_t boxA[3] = {BK, BM, 1};
    {
        const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Tb, (cuuint64_t)B};
        const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)Tb * K * 2};
        if (!pg_encode(&mB, b_src, 3, dims, strides, boxA)) return cudaErrorInvalidValue;
    }
    if (Ta > 0) {
        const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)Ta, (cuuint64_t)B};
        const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)Ta * K * 2};
        if (!pg_encode(&mA, a_src, 3, dims, strides, boxA)) return cudaErrorInvalidValue;
    } else {
        mA = mB;  // no memory rows: every row tile comes from b_src
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {BK, BN};
        if (!pg_encode(&mW, w, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    PgParams p;
    p.B = B;
    p.Ta = Ta;
    p.Tb = Tb;
    p.K = K;
    p.N = N;
    p.d = d;
    p.H = H;
    p.dh = dh;
    p.T_out = T_out;
    p.plain = plain;
    p.n_rt = (Ta + Tb) / BM;
    p.n_nt = N / BN;
    const long long tiles = (long long)B * p.n_rt * p.n_nt;
    if (tiles <= 0 || tiles > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    p.n_tiles = (int)tiles;
    p.out[0] = static_cast<__nv_bfloat16*>(out0);
    p.out[1] = static_cast<__nv_bfloat16*>(out1);
    p.out[2] = static_cast<__nv_bfloat16*>(out2);
    p.status = status;
    const int grid = p.n_tiles < pg_num_sms() ? p.n_tiles : pg_num_sms();
    proj_gemm_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(mA, mB, mW, p);
    return cudaGetLastError();
}

}  // namespace txl
