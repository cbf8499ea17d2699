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
// One launch may carry up to three GEMMs (q from h, k|v from [mem; h], and r
// from the position embedding) dealt from one tile list, so the smaller ones
// do not leave partial rounds (or, for r, a launch) of their own.
// One CTA per SM walks output tiles of 128 rows x 256 columns; K (= d) is
// streamed in 64-element steps through a 4-stage TMA ring (A tile 16 KB, B tile
// 32 KB, 128B swizzle).  Roles (384 threads): warp 0 lane 0 issues the TMA
// loads, warp 1 issues the MMAs (whole warp, one elected lane: M=128, N=256,
// K=16 per instruction into a TMEM accumulator), warps 4-11 drain the
// accumulator (one row per thread; warps w and w+4 split the 256 columns) to
// bf16, with the optional bias / ReLU / residual epilogue, and write it by
// TMA stores of staged 64-column slices.  Two accumulators of
// 256 columns let the epilogue of one tile overlap the MMAs of the next.
// Every wait is bounded (1 s) and reports through the device status word.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "proj_gemm.h"
#include "txl_device.cuh"

namespace txl {

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2,
                                             int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];\n\t"
        "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// the issuing thread's bulk stores have read / completed
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

namespace pg {
constexpr int BM = 128;     // rows per tile (TMEM lanes)
constexpr int BK = 64;      // K per stage: one 128-byte swizzle row of bf16
constexpr int NTHREADS = 384;  // warp 0 TMA, 1 MMA, 2-3 idle, 4-11 epilogue
constexpr uint32_t SZ_A = BM * BK * 2;  // 16 KB
constexpr uint32_t OFF_A = 0;
constexpr int MAX_STAGES = 6;

// Tile width BN (MMA N): 256 for the projections and wide outputs; 128 when
// the 256-wide tiles would leave most SMs with one tile and some with two.
template <int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    // measured at base512: 4 stages of 48 KB with one staged output slice per
    // epilogue warp beat 3 stages with two (q/k/v 28.3 -> 26.6 us): the MMAs
    // wait on the TMA loads, so bytes in flight count; 128-column tiles want 6
    static constexpr int STAGES = BN_ == 256 ? 4 : 6;
    static constexpr uint32_t SZ_B = BN_ * BK * 2;   // 32 or 16 KB
    static constexpr uint32_t OFF_B = OFF_A + STAGES * SZ_A;
    // output staging: each of the 8 epilogue warps stages one 64-column slice
    // of its 32 rows at a time (4 KB, 128-byte rows, 128-byte swizzle) and
    // waits until the slice's TMA store has read it before staging the next
    static constexpr uint32_t OFF_STG = OFF_B + STAGES * SZ_B;
    static constexpr uint32_t OFF_BAR = OFF_STG + 8 * 4096;  // one 64-column slice per warp
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t TMEM_COLS = 2 * BN_;  // two accumulators
    static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN_, 0);
    static_assert(SMEM_BYTES <= 232448, "shared memory budget of one sm_103a CTA");
    static_assert(STAGES <= MAX_STAGES, "barrier arrays");
};
}  // namespace pg

// One GEMM of the launch: per batch row, Ta rows of source a (the memory)
// then Tb rows of source b (current), times the problem's weights.
struct PgProblem {
    int B;          // batch rows of the problem
    int plain;      // 1: outputs are [rows, d] row-major (no head split)
    int Ta, Tb;     // rows per batch from source a, then source b (Ta a multiple of BM)
    int a_start;    // source a is a ring: logical row t is stored at row (a_start + t) % Ta
    int N;          // output columns (a multiple of BN)
    int T_out;      // rows per (batch, head) of the outputs
    int n_rt, n_nt, tiles;
    __nv_bfloat16* out[3];  // output column c -> tensor c / d
};

constexpr int kMaxProblems = 3;

struct PgParams {
    int K;          // reduction length (= d)
    int d, H, dh;   // output column c -> head (c % d) / dh, element c % dh
    int n_tiles;    // tiles of problem 0, then of problem 1, then of problem 2
    PgProblem pr[kMaxProblems];
    int* status;
    // plain outputs only: out = act(acc + bias[col]) + resid (resid laid
    // out like the output); null / 0 to skip
    const __nv_bfloat16* bias;
    const __nv_bfloat16* resid;
    int relu;
};

// Input tensor maps of problem g: source a, source b, weights.
struct PgIn {
    CUtensorMap m[kMaxProblems][3];
};

// Output tensor maps: problem g, output tensor o, viewed as (element of a
// 64-column slice, row t, slice (head, or 64-column chunk of a row-major
// output), batch row b); box 64 x 32 rows.
struct PgOut {
    CUtensorMap m[kMaxProblems][3];
};

struct PgShared {
    uint64_t full[pg::MAX_STAGES];
    uint64_t empty[pg::MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Tile w of the launch: problem 0's tiles, then problem 1's, then 2's; within
// a problem the column tile runs fastest, then the row tile, then the batch row.
template <int BN>
__device__ __forceinline__ int pg_tile(const PgParams& p, int w, int& b, int& t0, int& n0) {
    int g = 0;
    if (w >= p.pr[0].tiles) {
        w -= p.pr[0].tiles;
        g = 1;
        if (w >= p.pr[1].tiles) {
            w -= p.pr[1].tiles;
            g = 2;
        }
    }
    const PgProblem& pr = p.pr[g];
    const int nt = w % pr.n_nt, rest = w / pr.n_nt;
    n0 = nt * BN;
    t0 = (rest % pr.n_rt) * pg::BM;
    b = rest / pr.n_rt;
    return g;
}

template <int BN_>
__global__ void __launch_bounds__(pg::NTHREADS, 1)
proj_gemm_kernel(const __grid_constant__ PgIn inm, const __grid_constant__ PgOut outm, const PgParams p) {
    using namespace pg;
    using C = Cfg<BN_>;
    constexpr int BN = C::BN, STAGES = C::STAGES;
    constexpr uint32_t SZ_B = C::SZ_B, OFF_B = C::OFF_B, OFF_BAR = C::OFF_BAR, TMEM_COLS = C::TMEM_COLS,
                       IDESC = C::IDESC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    PgShared* sh = reinterpret_cast<PgShared*>(smem + OFF_BAR);
    const uint32_t s_base = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ksteps = p.K / BK;
    // programmatic stream serialisation: the next kernel may launch now; this
    // one waits for the previous kernel of the stream before any global access
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

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
            mbar_init(&sh->acc_empty[a], 8);  // one arrival per epilogue warp
        }
        mbar_init(&sh->drain, 1);
        sh->abort = 0;
        fence_mbar_init();
        for (int g = 0; g < kMaxProblems; ++g)
            if (p.pr[g].tiles > 0)
                for (int m = 0; m < 3; ++m) tma_prefetch_desc(&inm.m[g][m]);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            bool ok = true;
            int c = 0;  // loads issued into the ring
            for (int w = blockIdx.x; ok && w < p.n_tiles; w += gridDim.x) {
                int b, t0, n0;
                const int g = pg_tile<BN>(p, w, b, t0, n0);
                const int Ta = p.pr[g].Ta;
                // a row tile lies wholly in one source (Ta is a multiple of BM)
                const CUtensorMap* mA = t0 < Ta ? &inm.m[g][0] : &inm.m[g][1];
                // a_start and t0 are multiples of BM, so a ring tile never wraps
                const int ta = t0 < Ta ? (t0 + p.pr[g].a_start) % Ta : t0 - Ta;
                const CUtensorMap* mW = &inm.m[g][2];
                for (int k = 0; k < ksteps; ++k, ++c) {
                    const int s = c % STAGES;
                    if (c >= STAGES && !mbar_wait(&sh->empty[s], ((c / STAGES) & 1) ^ 1,
                                                  kDevTimeoutProducer, abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&sh->full[s], SZ_A + SZ_B);
                    tma_load_4d(smem + OFF_A + s * SZ_A, mA, &sh->full[s], 0, ta, k, b);
                    tma_load_2d(smem + OFF_B + s * SZ_B, mW, &sh->full[s], k * BK, n0);
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
        const int chalf = (warp - 4) >> 2;  // columns (BN / 2) chalf .. of the tile
        constexpr int CPW = BN / 64;         // 32-column chunks per epilogue warp
        const int row = wq * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t stg = s_base + C::OFF_STG + (uint32_t)(warp - 4) * 4096;
        bool store_pending = false;  // lane 0: this warp's last stores may still read the staging
        bool ok = true;
        int j = 0;
        for (int w = blockIdx.x; ok && w < p.n_tiles; w += gridDim.x, ++j) {
            const int acc = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&sh->acc_full[acc], (j >> 1) & 1,
                                                   kDevTimeoutSoftmax, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            int b, t0, n0;
            const int g = pg_tile<BN>(p, w, b, t0, n0);
            const PgProblem& pr = p.pr[g];
            const int t = t0 + row;
#pragma unroll 1
            for (int cc = CPW * chalf; cc < CPW * chalf + CPW; ++cc) {
                if ((cc & 1) == 0) {
                    if (store_pending) {
                        bulk_wait_read();  // the previous slice has been read
                        store_pending = false;
                    }
                    __syncwarp();
                }
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + acc * BN + 32 * cc, v);
                tmem_wait_ld();
                if (cc == CPW * chalf + CPW - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
                }
                const int n = n0 + 32 * cc;
                const int o = n / p.d, nd = n - o * p.d;
                __nv_bfloat16* const base = o == 0 ? pr.out[0] : (o == 1 ? pr.out[1] : pr.out[2]);
                __nv_bfloat16* dst;
                if (pr.plain) {
                    dst = base + ((size_t)b * pr.T_out + t) * p.d + nd;
                } else {
                    const int head = nd / p.dh, e = nd - head * p.dh;
                    dst = base + (((size_t)b * p.H + head) * pr.T_out + t) * p.dh + e;
                }
                if (p.bias || p.relu || p.resid) {
                    // the row-major epilogue of a plain Linear: bias, ReLU, residual
                    float f[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) f[x] = __uint_as_float(v[x]);
                    // bias: d columns; residual: laid out like the plain output [B, T_out, d]
                    if (p.bias && TXL_BOUNDS(n + 32 <= p.d, 601, n)) {
                        const uint4* b4 = reinterpret_cast<const uint4*>(p.bias + n);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 w4 = __ldg(b4 + q);
                            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w4);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 bf = __bfloat1622float2(h2[e]);
                                f[8 * q + 2 * e] += bf.x;
                                f[8 * q + 2 * e + 1] += bf.y;
                            }
                        }
                    }
                    if (p.relu) {
#pragma unroll
                        for (int x = 0; x < 32; ++x) f[x] = fmaxf(f[x], 0.f);
                    }
                    if (p.resid && TXL_BOUNDS((dst - base) >= 0 && (dst - base) + 32 <= (long long)pr.B * pr.T_out * p.d,
                                              602, dst - base)) {
                        const uint4* r4 = reinterpret_cast<const uint4*>(p.resid + (dst - base));
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 w4 = __ldg(r4 + q);
                            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w4);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 rf = __bfloat1622float2(h2[e]);
                                f[8 * q + 2 * e] += rf.x;
                                f[8 * q + 2 * e + 1] += rf.y;
                            }
                        }
                    }
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = __float_as_uint(f[x]);
                }
                // stage the 32 columns in the warp's 64-column slice (row = lane,
                // 16-byte chunk c at c ^ (lane & 7)); a full slice goes out as one
                // TMA store of 32 rows
                const uint32_t slice = stg;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c16 = 4 * (cc & 1) + q;
                    if (TXL_BOUNDS(slice + lane * 128 + ((c16 ^ (lane & 7)) << 4) + 16 <= s_base + C::SMEM_BYTES &&
                                       slice >= s_base,
                                   603, (long long)slice - s_base))
                    st_shared_v4(slice + lane * 128 + ((c16 ^ (lane & 7)) << 4),
                                 pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                }
                if (cc & 1) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int ns = n - 32;  // the slice's first column
                        const int os = ns / p.d, nds = ns - os * p.d;
                        tma_store_4d(&outm.m[g][os], slice, 0, t0 + 32 * wq, pr.plain ? nds / 64 : nds / p.dh, b);
                        store_pending = true;
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // the stores complete before the CTA exits
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
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch with programmatic stream serialisation (the kernel waits for the
// previous kernel of the stream before its first global access).
template <typename Kern>
static cudaError_t launch_pg_pdl(Kern kern, int grid, uint32_t smem, cudaStream_t stream, const PgIn& inm,
                                 const PgOut& outm, const PgParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(pg::NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, inm, outm, p);
}

// Output map of one bf16 tensor: heads [B, H, T, dh] (dh = 64) or row-major
// [B, T, width], as (element of a 64-column slice, row, slice, batch).
static bool pg_encode_out(CUtensorMap* map, void* base, int B, int T, int width, int heads_layout) {
    const int slices = width / 64;
    const cuuint64_t dims[4] = {64, (cuuint64_t)T, (cuuint64_t)slices, (cuuint64_t)B};
    const cuuint64_t row = heads_layout ? 128 : (cuuint64_t)width * 2;
    const cuuint64_t slice = heads_layout ? (cuuint64_t)T * 128 : 128;
    const cuuint64_t strides[3] = {row, slice, (cuuint64_t)T * width * 2};
    const cuuint32_t box[4] = {64, 32, 1, 1};
    return pg_encode(map, base, 4, dims, strides, box);
}

static int pg_num_sms() { return current_sm_count(); }

// (declared in proj_gemm.h)
cudaError_t launch_proj_gemm(const ProjGemm* gm, int n_gemm, int B, int K, int d, int H, int dh,
                             int plain, int* status, cudaStream_t stream) {
    using namespace pg;
    using C = Cfg<256>;
    constexpr int BN = C::BN;
    static PerDeviceOnce attrs;
    {
        const cudaError_t e = attrs.run([] {
            return cudaFuncSetAttribute(proj_gemm_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
        });
        if (e != cudaSuccess) return e;
    }
    if (n_gemm < 1 || n_gemm > kMaxProblems) return cudaErrorInvalidValue;
    PgIn inm;  // per problem: source a, source b, weights
    PgOut outm;
    PgParams p;
    p.K = K;
    p.d = d;
    p.H = H;
    p.dh = dh;
    p.status = status;
    p.bias = nullptr;
    p.resid = nullptr;
    p.relu = 0;
    // Both layouts as one 4-D view (element, row t, 64-column chunk k, batch
    // row b), so the kernel loads chunk k of rows t0.. with coordinates
    // (0, t0, k, b) either way.
    auto encode_src = [&](CUtensorMap* map, const void* src, int T, int heads, int Bp) {
        const cuuint64_t dims[4] = {(cuuint64_t)BK, (cuuint64_t)T, (cuuint64_t)(K / BK), (cuuint64_t)Bp};
        const cuuint64_t row = heads ? (cuuint64_t)BK * 2 : (cuuint64_t)K * 2;
        const cuuint64_t chunk = heads ? (cuuint64_t)T * BK * 2 : (cuuint64_t)BK * 2;
        const cuuint64_t strides[3] = {row, chunk, (cuuint64_t)T * K * 2};
        const cuuint32_t box[4] = {BK, BM, 1, 1};
        return pg_encode(map, src, 4, dims, strides, box);
    };
    long long total = 0;
    for (int g = 0; g < kMaxProblems; ++g) {
        const ProjGemm& q = gm[g < n_gemm ? g : 0];
        const int Bp = q.B > 0 ? q.B : B;
        const int plain_g = q.plain >= 0 ? q.plain : plain;
        if (!encode_src(&inm.m[g][1], q.b_src, q.Tb, q.b_heads, Bp)) return cudaErrorInvalidValue;
        if (q.Ta > 0) {
            if (!encode_src(&inm.m[g][0], q.a_src, q.Ta, q.a_heads, Bp)) return cudaErrorInvalidValue;
        } else {
            inm.m[g][0] = inm.m[g][1];  // no memory rows: every row tile comes from b_src
        }
        {
            const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)q.N};
            const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
            const cuuint32_t box[2] = {BK, BN};
            if (!pg_encode(&inm.m[g][2], q.w, 2, dims, strides, box)) return cudaErrorInvalidValue;
        }
        PgProblem& pr = p.pr[g];
        pr.B = Bp;
        pr.plain = plain_g;
        pr.Ta = q.Ta;
        pr.Tb = q.Tb;
        pr.a_start = q.a_start;
        pr.N = q.N;
        pr.T_out = q.T_out;
        pr.n_rt = (q.Ta + q.Tb) / BM;
        pr.n_nt = q.N / BN;
        const long long tiles = g < n_gemm ? (long long)Bp * pr.n_rt * pr.n_nt : 0;
        pr.tiles = (int)(tiles > 0x7FFFFFFFll ? 0 : tiles);
        total += tiles;
        for (int o = 0; o < 3; ++o) pr.out[o] = static_cast<__nv_bfloat16*>(q.out[o]);
        // one map per output tensor of the problem (N / d of them); unused
        // entries repeat the first
        const int n_out = q.N / d;
        for (int o = 0; o < 3; ++o) {
            if (o < n_out) {
                if (!pg_encode_out(&outm.m[g][o], q.out[o], Bp, q.T_out, d, !plain_g)) return cudaErrorInvalidValue;
            } else {
                outm.m[g][o] = outm.m[g][0];
            }
        }
    }
    if (total <= 0 || total > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    p.n_tiles = (int)total;
    const int grid = p.n_tiles < pg_num_sms() ? p.n_tiles : pg_num_sms();
    return launch_pg_pdl(proj_gemm_kernel<256>, grid, C::SMEM_BYTES, stream, inm, outm, p);
}

// A plain Linear over rows of x (layout 0: [B, T, K]; 1: [B, K / 64, T, 64]):
// out [B, T, N] = relu?(x W^T + bias) + resid, all bf16, fp32 accumulation.
template <int BN_>
static cudaError_t launch_linear_bn(const void* x, int x_heads, int B, int T, int K, const void* w, int N,
                                   const void* bias, const void* resid, int relu, void* out, int* status,
                                   cudaStream_t stream) {
    using namespace pg;
    using C = Cfg<BN_>;
    constexpr int BN = C::BN;
    static PerDeviceOnce attrs;
    {
        const cudaError_t e = attrs.run([] {
            return cudaFuncSetAttribute(proj_gemm_kernel<BN_>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
        });
        if (e != cudaSuccess) return e;
    }
    PgIn inm;
    CUtensorMap* maps = inm.m[0];
    {
        const cuuint64_t dims[4] = {(cuuint64_t)BK, (cuuint64_t)T, (cuuint64_t)(K / BK), (cuuint64_t)B};
        const cuuint64_t row = x_heads ? (cuuint64_t)BK * 2 : (cuuint64_t)K * 2;
        const cuuint64_t chunk = x_heads ? (cuuint64_t)T * BK * 2 : (cuuint64_t)BK * 2;
        const cuuint64_t strides[3] = {row, chunk, (cuuint64_t)T * K * 2};
        const cuuint32_t box[4] = {BK, BM, 1, 1};
        if (!pg_encode(&maps[0], x, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {BK, BN};
        if (!pg_encode(&maps[2], w, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    maps[1] = maps[0];
    PgParams p;
    p.K = K;
    p.d = N;   // one output, row-major [B, T, N]
    p.H = 1;
    p.dh = N;
    p.status = status;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.resid = static_cast<const __nv_bfloat16*>(resid);
    p.relu = relu;
    PgProblem& pr = p.pr[0];
    pr.B = B;
    pr.plain = 1;
    pr.Ta = 0;
    pr.Tb = T;
    pr.a_start = 0;
    pr.N = N;
    pr.T_out = T;
    pr.n_rt = T / BM;
    pr.n_nt = N / BN;
    const long long tiles = (long long)B * pr.n_rt * pr.n_nt;
    if (tiles <= 0 || tiles > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    pr.tiles = (int)tiles;
    pr.out[0] = static_cast<__nv_bfloat16*>(out);
    pr.out[1] = pr.out[2] = nullptr;
    PgOut outm;
    if (!pg_encode_out(&outm.m[0][0], out, B, T, N, 0)) return cudaErrorInvalidValue;
    for (int i = 0; i < kMaxProblems * 3; ++i) (&outm.m[0][0])[i] = outm.m[0][0];
    for (int g = 1; g < kMaxProblems; ++g) {
        for (int m = 0; m < 3; ++m) inm.m[g][m] = inm.m[0][m];
        p.pr[g] = pr;
        p.pr[g].tiles = 0;
    }
    p.n_tiles = (int)tiles;
    const int grid = p.n_tiles < pg_num_sms() ? p.n_tiles : pg_num_sms();
    return launch_pg_pdl(proj_gemm_kernel<BN_>, grid, C::SMEM_BYTES, stream, inm, outm, p);
}

// 256-column tiles unless that leaves fewer than two tiles per SM (then
// 128-column tiles: twice the tiles, each half the work, for a better fill).
cudaError_t launch_linear(const void* x, int x_heads, int B, int T, int K, const void* w, int N,
                          const void* bias, const void* resid, int relu, void* out, int* status,
                          cudaStream_t stream) {
    const long long wide = (long long)B * (T / pg::BM) * (N / 256);
    if (wide < 2ll * pg_num_sms())
        return launch_linear_bn<128>(x, x_heads, B, T, K, w, N, bias, resid, relu, out, status, stream);
    return launch_linear_bn<256>(x, x_heads, B, T, K, w, N, bias, resid, relu, out, status, stream);
}

TXL_BOUNDS_READER(bounds_word_proj_gemm)

}  // namespace txl
