// Fused Transformer-XL relative attention, bf16 in / fp32 accumulate, on the
// sm_103a tensor cores (tcgen05 + TMEM), with TMA-staged K, V and R tiles.
//
// Unit of work ("item"): one (batch row b, head h, query tile of 128 rows
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
// 64t) needs the 191 R rows base+64t .. base+64t+190 (base = L-i0-128): three
// 64-row "slots" g = t, t+1, t+2 of the sequence base+64g.  Consecutive tiles
// share two slots, so the key tiles go out in pairs (2p, 2p+1) and each pair
// computes only its two newest slots 2p+2, 2p+3 (the first pair slots 0-3),
// one 128-row R box, into a 4-slot ring of TMEM columns: the position MMA does
// the algorithmic work plus at most one slot per item.  Row ii of the band, read from band
// column 127-ii onward, is the shifted position term: the pad / reshape /
// slice of the pages is never performed and no L x (M+L) score matrix exists.
// R rows outside [0, M+L) are zero-filled by TMA and only land on masked
// entries.
//
// Persistent schedule.  One CTA per SM walks its items (longest query tiles
// first, snake order over CTAs).  The TMA producer and the MMA issuer stream
// across item boundaries; (q+u)c / (q+v)c are double-buffered so the next
// item's scores can start while the current item is finished and stored.
//
// Roles (384 threads; warp w runs on SM sub-partition w % 4):
//   warps 0-7  two softmax groups of 128 threads (one query row per thread;
//              group 0 = warps 0, 2, 5, 7, group 1 = warps 1, 3, 4, 6);
//              group g takes the item's key tiles t = g (mod 2),
//              keeps its own running max, sum and O accumulator, and the two
//              partial results are merged per item
//   warp 8     TMEM allocation; issues the score MMAs (AC and position slots)
//   warp 9     lane 0 initialises the barriers, issues the first item's
//              loads before the block synchronises, then all TMA loads
//              (128-row boxes: per-SM TMA throughput grows with the box
//              size) and L2 prefetches
//   warp 10    issues the P V MMAs
//   warp 11    prepares the score MMAs' A operands of each item after the
//              first: loads the raw q tile by TMA into both slots of the
//              item's Q buffer and rewrites them in place as (q+u)c and
//              (q+v)c (the softmax groups do the first item's)
// The score and P V chains are issued from different sub-partitions so that
// neither waits behind the other or behind the softmax warps' instruction
// streams.
//
// TMEM columns: O0 0-63, O1 64-127, AC0 128-191, AC1 192-255, position ring
// 256-511.  Shared memory: (q+u)c,(q+v)c x2 (each first filled with the raw q
// tile by TMA, then rewritten in place), P x2, K/V ring, R ring.  At the end
// of an item each softmax warp stages its 32 rows of its group's 32 output
// columns in its own quarter of the P buffer and writes them with one TMA
// store.  A group's P
// buffer is also the scratch of its per-row shift: after the group's previous
// P V finished and before the new P is written, each warp moves its rows'
// band windows through its 4 KB quarter of it, two band columns (c, c+32)
// per 32-bit word as f16x2 (the position term is rounded to f16 there and
// added to the f32 content term in f32).
//
// Registers: warps 8-11 give up registers (setmaxnreg) so that each softmax
// thread can hold its row's 64 content terms and 96 band columns at once.
//
// Ordering facts relied on: tcgen05.mma operations from one thread execute in
// issue order, and a tcgen05.commit arrives only when every MMA issued before
// it by the same thread has completed.
//
// Every mbarrier wait is bounded (1 s); on expiry the CTA records a status,
// drains its in-flight copies and MMAs, frees TMEM and exits.  The named
// barriers of the per-item merge (bar 1, all 256 softmax threads) have no
// time limit: one snapshot of the abort flag taken between the first two
// decides, for all 256 threads at once, whether the merge and the next item
// run.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_tc_common.cuh"
#include "txl_device.cuh"

namespace txl {

namespace tc {
constexpr int BM = 128;        // query rows per item (TMEM lanes)
constexpr int BN = 64;         // keys per tile
constexpr int DH = 64;         // head dim: one 128-byte swizzle row
constexpr int SLOT = 64;       // R rows per position slot
constexpr int RING = 4;        // position slots held in TMEM
#ifndef TXL_KV_STAGES
#define TXL_KV_STAGES 3
#endif
#ifndef TXL_R_STAGES
#define TXL_R_STAGES 2
#endif
#ifndef TXL_PREFETCH
#define TXL_PREFETCH 2
#endif
constexpr int KV_STAGES = TXL_KV_STAGES;  // K/V ring: each stage holds two key tiles
constexpr int R_STAGES = TXL_R_STAGES;    // R ring: each box holds two position slots
constexpr int PREFETCH = TXL_PREFETCH;    // K/V stages warmed into L2 ahead of their load
static_assert(KV_STAGES >= 2 && R_STAGES >= 2, "the MMA order needs two stages of each ring");
constexpr int NTHREADS = 384;

constexpr uint32_t SZ_T = BN * DH * 2;      //  8 KB: one 64-row tile
constexpr uint32_t SZ_BOX = 2 * SZ_T;       // 16 KB: one 128-row TMA box
constexpr uint32_t SZ_Q = BM * DH * 2;      // 16 KB
constexpr uint32_t OFF_Q = 0;               // buffer b: (q+u)c at +32K*b, (q+v)c at +32K*b+16K
constexpr uint32_t OFF_P = OFF_Q + 4 * SZ_Q;          // P of group g at +16K*g; merge exchange
constexpr uint32_t OFF_KV = OFF_P + 2 * SZ_Q;         // stage s: K box, V box
constexpr uint32_t OFF_R = OFF_KV + KV_STAGES * 2 * SZ_BOX;
constexpr uint32_t OFF_BAR = OFF_R + R_STAGES * SZ_BOX;
constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one sm_103a CTA");

constexpr uint32_t COL_O = 0;       // + 64 * group
constexpr uint32_t COL_AC = 128;    // + 64 * group
constexpr uint32_t COL_RING = 256;  // + 64 * slot
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t IDESC_N64 = idesc_bf16_f32(128, 64, 0);    // K-major B: one key tile
constexpr uint32_t IDESC_N128 = idesc_bf16_f32(128, 128, 0);  // K-major B: a K or R box
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
    int n_items;       // (b, h, query tile) items
    int nsplit;        // key splits per item (1: the kernel writes the output)
    int n_units;       // n_items * nsplit work units
    float* ws_o;       // nsplit > 1: unnormalised O of each unit, [unit][128][64]
    float2* ws_ml;     // nsplit > 1: (m, l) of each unit's rows, [unit][128]
    float scale_log2;  // scale * log2(e), folded into q+u and q+v
    int inject;        // 1: withhold the first score-ready signal (timeout test)
    int* status;       // device status word
    int lo_shift;      // keys j < i + 1 - lo_shift are masked too (same_length; 1 << 30: none)
    float* lse;        // non-null: per-row log2-sum-exp of the scores, [B*H][L]
};

struct TcShared {
    uint64_t kv_full[tc::KV_STAGES];
    uint64_t kv_empty[tc::KV_STAGES];
    uint64_t r_full[tc::R_STAGES];
    uint64_t r_empty[tc::R_STAGES];
    uint64_t q_ready;     // (q+u)c and (q+v)c of the next item are in shared memory
    uint64_t q_full;      // the raw q tile of the next item landed in both slots
    uint64_t s_full[2];   // scores of the group's next tile are in TMEM
    uint64_t s_free[2];   // the group has read them into registers
    uint64_t p_full[2];   // the group's P tile is in shared memory
    uint64_t pv_done[2];  // the group's last P V MMA finished
    uint64_t o_done;      // every MMA of the item finished: O may be read
    uint64_t o_free;      // the merge has read both O accumulators
    uint64_t drain;
    uint64_t q_free;      // the first score pair of an item (and all before it) completed
    uint32_t tmem_base;
    int abort;
    int merge_abort;      // the abort flag as seen once per item by the merge
};

// One work unit and the quantities every role derives from it: the key tiles
// t0 .. t0+ntiles-1 of one (b, h, query tile) item (all of them unless the
// item is split over several units).
struct Item {
    int bh, h, i0, t0, ntiles, rbase, unit;
};

// k-th unit of this CTA: items are numbered longest query tile first, the
// splits of an item are adjacent, and units are dealt to CTAs in snake order
// (rounds alternate direction) to even out the load.  A split takes a
// contiguous range of tile pairs, so t0 is even.
template <bool SPLIT, bool LOWER>
__device__ __forceinline__ bool item_of(const TcParams& p, int k, Item& it) {
    const int G = gridDim.x, c = blockIdx.x;
    const int w = k * G + ((k & 1) ? (G - 1 - c) : c);  // below 2^31: checked at launch
    if (w >= p.n_units) return false;
    int witem = w, sp = 0;
    if constexpr (SPLIT) {
        witem = w / p.nsplit;
        sp = w - witem * p.nsplit;
    }
    const int n_bh = p.B * p.H;
    const int qq = witem / n_bh;
    const int qt = p.n_qtiles - 1 - qq;
    it.bh = witem - qq * n_bh;
    it.h = it.bh % p.H;
    it.i0 = qt * tc::BM;
    const int rows_valid = min(tc::BM, p.L - it.i0);
    const int kmax = p.M + it.i0 + rows_valid - 1;  // last key any row of the tile sees
    const int all = kmax / tc::BN + 1;
    // first key any row of the tile sees (same_length), rounded down to a
    // tile pair: tiles below it are skipped
    int tlo = 0;
    if constexpr (LOWER) {
        const int jmin = it.i0 + 1 - p.lo_shift;
        tlo = jmin > 0 ? ((jmin / tc::BN) & ~1) : 0;
    }
    it.t0 = tlo;
    it.ntiles = all - tlo;
    if constexpr (SPLIT) {
        const int pairs = (all - tlo + 1) >> 1;
        const int lo = pairs * sp / p.nsplit, hi = pairs * (sp + 1) / p.nsplit;
        it.t0 = tlo + 2 * lo;
        it.ntiles = min(tlo + 2 * hi, all) - it.t0;
    }
    it.rbase = p.L - it.i0 - tc::BM + tc::SLOT * it.t0;  // R row of the unit's slot 0
    it.unit = w;
    return true;
}

// Position slots an item occupies in the ring: slots 0 .. ntiles+1 are read,
// rounded up to an even count so that every item starts on an even global
// slot and each score MMA writes two adjacent slots (one R box of 128 rows).
__device__ __forceinline__ int slots_of(int ntiles) { return 2 * (((ntiles + 1) >> 1) + 1); }

// Bounds-checked builds: a shared-memory access of `bytes` at `addr` stays
// inside this CTA's dynamic shared memory.
#define TXL_SMEM_IN(addr, bytes, site) \
    TXL_BOUNDS((addr) >= s_base && (addr) + (bytes) <= s_base + tc::SMEM_BYTES, (site), (long long)(addr) - s_base)

// SPLIT: the units are key splits of items and write partial results (see
// attn_combine_kernel); otherwise every unit is a whole item.  LOWER: the
// same_length lower key bound is applied (tiles below it skipped, keys below
// it masked).
template <bool SPLIT, bool LOWER>
__global__ void __launch_bounds__(tc::NTHREADS, 1)
attn_tc_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmR,
                    const __grid_constant__ CUtensorMap tmO, const TcParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    TcShared* sh = reinterpret_cast<TcShared*>(smem + OFF_BAR);
    const uint32_t s_base = smem_u32(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // Launched with programmatic stream serialisation: the next kernel of the
    // stream may start its prologue while this grid's CTAs finish (none of
    // its CTAs fits beside one of these, so it only takes SMs as they free
    // up); every global access here comes after the wait for the previous
    // kernel of the stream to complete.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 8) {
        tmem_alloc(&sh->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    // The TMA producer thread initialises the barriers and issues the first
    // item's loads (its q tile, K/V stage 0, R boxes 0 and 1) before the block
    // synchronises, so that their DRAM latency overlaps the prologue.
    int pre_kv = 0, pre_r = 0;  // loads of item 0 issued here
    if (warp == 9 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmR);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(&sh->kv_full[s], 1);
            mbar_init(&sh->kv_empty[s], 1);
        }
        for (int s = 0; s < R_STAGES; ++s) {
            mbar_init(&sh->r_full[s], 1);
            mbar_init(&sh->r_empty[s], 1);
        }
        // softmax-side barriers count warps: one elected lane per warp arrives
        mbar_init(&sh->q_ready, 8);  // 8 warp arrivals, or one arrival counting 8
        mbar_init(&sh->q_full, 1);
        mbar_init(&sh->q_free, 1);
        for (int g = 0; g < 2; ++g) {
            mbar_init(&sh->s_full[g], 1);
            mbar_init(&sh->s_free[g], 4);
            mbar_init(&sh->p_full[g], 4);
            mbar_init(&sh->pv_done[g], 1);
        }
        mbar_init(&sh->o_done, 1);
        mbar_init(&sh->o_free, 8);
        mbar_init(&sh->drain, 2);  // one commit from each MMA issuer
        sh->abort = 0;
        fence_mbar_init();
        asm volatile("griddepcontrol.wait;" ::: "memory");
        Item it0;
        if (item_of<SPLIT, LOWER>(p, 0, it0)) {
            mbar_expect_tx(&sh->q_full, 2 * SZ_Q);
            tma_load_3d(smem + OFF_Q, &tmQ, &sh->q_full, 0, it0.i0, it0.bh);
            tma_load_3d(smem + OFF_Q + SZ_Q, &tmQ, &sh->q_full, 0, it0.i0, it0.bh);
            mbar_expect_tx(&sh->kv_full[0], 2 * SZ_BOX);
            tma_load_3d(smem + OFF_KV, &tmK, &sh->kv_full[0], 0, it0.t0 * BN, it0.bh);
            tma_load_3d(smem + OFF_KV + SZ_BOX, &tmV, &sh->kv_full[0], 0, it0.t0 * BN, it0.bh);
            pre_kv = 1;
            const int nrb = (it0.ntiles + 3) >> 1;
            for (; pre_r < 2 && pre_r < nrb; ++pre_r) {
                mbar_expect_tx(&sh->r_full[pre_r], SZ_BOX);
                tma_load_2d(smem + OFF_R + pre_r * SZ_BOX, &tmR, &sh->r_full[pre_r], it0.h * DH,
                            it0.rbase + SLOT * 2 * pre_r);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;
    // Register split: the softmax warpgroups hold a whole tile's scores and
    // band (160 values) at once.  Launched with 168 per thread (384 x 168 =
    // 64,512); 2 x 128 x 200 + 128 x 96 = 63,488 fits in that.
    if (warp >= 8)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
    else
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");

    if (warp < 8) {
        // ------------------------------------------------------ softmax groups
        // Groups {0, 2, 5, 7} and {1, 3, 4, 6}: each covers the four TMEM lane
        // quarters (warp w reads lanes 32 (w % 4) ..) and holds two of the four
        // lower warp ids the schedulers favour, so neither group lags by design
        const int grp = ((warp >> 2) ^ warp) & 1;
        const int wq = warp & 3;            // TMEM lane quarter
        const int ii = tid & 127;           // query row within the item
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t col_ac = COL_AC + 64 * grp;
        const uint32_t p_tile = s_base + OFF_P + grp * SZ_Q;
        // this warp's quarter of the group's P buffer doubles as the row-shift
        // scratch T[pos][lane] (word pos * 32 + lane) before P is written
        const uint32_t t_ld = p_tile + wq * 4096 + 4 * lane;
        const uint32_t t_st = t_ld - 128u * (uint32_t)(31 - lane);
        bool ok = true;

        Item cur;
        bool store_pending = false;  // lane 0: this warp's output box may still be being read
        int it_g = 0;      // tiles this group has processed (all items)
        int gbase = 0;     // global position-slot counter of the item's slot 0 (even)
        for (int k = 0; ok && item_of<SPLIT, LOWER>(p, k, cur); ++k) {
            if (k == 0) {
                // the first item's operands: the groups are idle until its first
                // scores, so they convert it themselves (warp 11 takes the rest);
                // its q tile was loaded in the prologue
                const uint4* brow = reinterpret_cast<const uint4*>((grp == 0 ? p.ub : p.vb) + (size_t)cur.h * DH);
                uint4 b4[8];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    b4[ch] = TXL_BOUNDS(cur.h < p.H, 401, cur.h) ? __ldg(brow + ch) : make_uint4(0, 0, 0, 0);
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->q_full, 0, kDevTimeoutSoftmax, abort, p.status));
                if (!ok && tid == 0) drain_wait(&sh->q_full, 0, p.status);
                if (ok) {
                    const uint32_t row = s_base + OFF_Q + grp * SZ_Q + ii * 128;
                    const float qscale = p.scale_log2;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint32_t a = row + ((ch ^ (ii & 7)) << 4);
                        float raw[4];
                        if (!TXL_SMEM_IN(a, 16, 402)) continue;
                        ld_shared_v4(a, raw);
                        const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(raw);
                        const __nv_bfloat162* bb = reinterpret_cast<const __nv_bfloat162*>(&b4[ch]);
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 qf = __bfloat1622float2(q2[e]);
                            const float2 bf = __bfloat1622float2(bb[e]);
                            w[e] = pack_bf16x2((qf.x + bf.x) * qscale, (qf.y + bf.y) * qscale);
                        }
                        st_shared_v4(a, w[0], w[1], w[2], w[3]);
                    }
                    fence_proxy_async_smem();
                    warp_arrive(&sh->q_ready);
                }
            }
            const int i = cur.i0 + ii;
            float m_run = -INFINITY;  // running max (log2 domain), may lag the true max by < 8
            float l_run = 0.f;
            int seen = 0;             // this group's tiles in this item
            for (int t = grp; t < cur.ntiles; t += 2) {
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->s_full[grp], it_g & 1,
                                                       kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
                tc_fence_after();
                if (it_g > 0) {
                    // the group's previous P V must be done before its P buffer
                    // is reused (shift scratch, then P) or O is rescaled
                    ok = __all_sync(0xffffffffu, mbar_wait(&sh->pv_done[grp], (it_g - 1) & 1,
                                                           kDevTimeoutSoftmax, abort, p.status));
                    if (!ok) break;
                    tc_fence_after();
                }
                const int j0 = (cur.t0 + t) * BN;
                // the diagonal crosses the tile, or (same_length) the lower bound
                // of the tile's last row lies past its first key
                const bool need_mask =
                    (j0 + BN - 1) > (p.M + cur.i0) || (LOWER && j0 < cur.i0 + BM - p.lo_shift);
                const int jlim = p.M + i - j0;       // keys jj > jlim are masked
                const int jlo = i + 1 - p.lo_shift - j0;  // and keys jj < jlo
                float sc[BN];
                {
                    // the tile's AC (64 columns) and band columns c0 .. c0+95,
                    // c0 = 96 - 32*wq: row ii's window starts at band column
                    // 127 - ii = c0 + (31 - lane).  Band column c lives in ring
                    // slot (global slot of t) + c/64 (item slot t + c/64 is
                    // global slot gbase + t + c/64).  One wait, then the
                    // scores are released to the next pair's MMAs.
                    uint32_t ac[BN], bw[96];
                    tmem_ld32(tmem + lane_off + col_ac, *reinterpret_cast<uint32_t(*)[32]>(&ac[0]));
                    tmem_ld32(tmem + lane_off + col_ac + 32, *reinterpret_cast<uint32_t(*)[32]>(&ac[32]));
#pragma unroll
                    for (int kc = 0; kc < 3; ++kc) {
                        const int c = 96 - 32 * wq + 32 * kc;
                        const uint32_t rc = COL_RING + 64 * ((gbase + t + (c >> 6)) & (RING - 1)) + (c & 63);
                        tmem_ld32(tmem + lane_off + rc, *reinterpret_cast<uint32_t(*)[32]>(&bw[32 * kc]));
                    }
                    tmem_wait_ld();
                    tc_fence_before();
                    warp_arrive(&sh->s_free[grp]);
                    // The shift moves band pairs (c, c+32) packed as f16x2, so
                    // one pass through the warp's scratch aligns both halves of
                    // the window: word K = (band c0+K, band c0+K+32), and
                    // position x of the shifted row is word (31 - lane) + x =
                    // the terms of keys x and x+32.  Half the shared-memory
                    // traffic of moving f32 values.  The f16 rounding changes
                    // the position term (already in log2 units: scale * log2 e
                    // is folded into q+v) by at most 2^-11 |BD|, relative
                    // rounding of an 11-bit significand; |BD| > 65504 would
                    // saturate, far beyond any softmax score that matters.
                    uint32_t hp[64];
#pragma unroll
                    for (int K = 0; K < 64; ++K)
                        hp[K] = pack_f16x2_sat(__uint_as_float(bw[K]), __uint_as_float(bw[K + 32]));
                    float win[32];
                    if (store_pending) {
                        // the previous item's output box has been read
                        bulk_wait_read();
                        store_pending = false;
                    }
                    __syncwarp();
                    if (!TXL_SMEM_IN(t_ld, 128 * 31 + 4, 403)) break;
                    st_shift_all<0>(31 - lane, t_st, *reinterpret_cast<uint32_t(*)[32]>(&hp[0]),
                                    *reinterpret_cast<uint32_t(*)[32]>(&hp[32]));
                    ld_shift_all<0>(t_ld, win);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const float2 s2 = add_h2_f32(__float_as_uint(win[x]), __uint_as_float(ac[x]),
                                                     __uint_as_float(ac[x + 32]));
                        sc[x] = s2.x;
                        sc[x + 32] = s2.y;
                    }
                }
                if (need_mask) {
#pragma unroll
                    for (int x = 0; x < BN; ++x)
                        if (x > jlim || (LOWER && x < jlo)) sc[x] = -INFINITY;
                }
                float tmax = -INFINITY;
#pragma unroll
                for (int x = 0; x < BN; x += 2) tmax = max3(tmax, sc[x], sc[x + 1]);
                // Conditional rescale: keep the running max unless the tile's max
                // exceeds it by more than the threshold (then p <= 2^threshold).
                const float m_new = (tmax > m_run + kRescaleThreshold) ? tmax : m_run;
                // A row may have seen no visible key yet in this group (m_new =
                // -inf): exponentiate against 0 instead, so every p is 0, not NaN.
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = ex2(m_run - m_use);
                if (seen > 0 && __any_sync(0xffffffffu, m_new != m_run)) {
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
                __syncwarp();  // every lane's scratch reads precede the P rows
                const float2 negm = make_float2(-m_use, -m_use);
                float2 rs = make_float2(0.f, 0.f);
#pragma unroll
                for (int c8 = 0; c8 < BN / 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x =
                            add2(make_float2(sc[c8 * 8 + 2 * e], sc[c8 * 8 + 2 * e + 1]), negm);
                        const float p0 = ex2(x.x), p1 = ex2(x.y);
                        rs = add2(rs, make_float2(p0, p1));
                        w[e] = pack_bf16x2(p0, p1);
                    }
                    if (TXL_SMEM_IN(p_tile + ii * 128 + ((c8 ^ (ii & 7)) << 4), 16, 404))
                        st_shared_v4(p_tile + ii * 128 + ((c8 ^ (ii & 7)) << 4), w[0], w[1], w[2], w[3]);
                }
                l_run = l_run * alpha + (rs.x + rs.y);
                m_run = m_new;
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&sh->p_full[grp]);
                ++it_g;
                ++seen;
            }
            // ---------------------------------------------- merge + store
            if (ok)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&sh->o_done, k & 1, kDevTimeoutSoftmax, abort, p.status));
            // Each group finishes half of the output columns (group g: 32g ..
            // 32g+31) from both accumulators, which its warps read straight from
            // TMEM; only the per-row (m, l) cross between the groups, through
            // the other group's P buffer (idle until that group's next tile, so
            // one barrier suffices).  l = -1 marks a group without a tile in
            // this item: its O is stale and is not read.  The second barrier
            // keeps every P write of the next tiles behind all (m, l) reads.
            {
                float* ml_out = reinterpret_cast<float*>(smem + OFF_P + (grp ^ 1) * SZ_Q);
                if (TXL_SMEM_IN(smem_u32(ml_out + 2 * ii), 8, 405)) {
                    ml_out[2 * ii] = seen ? m_run : -INFINITY;
                    ml_out[2 * ii + 1] = seen ? l_run : -1.f;
                }
            }
            // both groups reach these barriers on every path (ok is warp-uniform)
            asm volatile("bar.sync 1, 256;" ::: "memory");
            float mo, lo;
            {
                const float* ml_in = reinterpret_cast<const float*>(smem + OFF_P + grp * SZ_Q);
                mo = -INFINITY;
                lo = -1.f;
                if (TXL_SMEM_IN(smem_u32(ml_in + 2 * ii), 8, 406)) {
                    mo = ml_in[2 * ii];
                    lo = ml_in[2 * ii + 1];
                }
            }
            // One snapshot of the abort flag decides for all 256 threads, so
            // that either every softmax warp runs the merge (with its group
            // barriers) and the next item, or none does.  A warp whose wait
            // failed set the flag before it reached the first barrier.
            if (tid == 0) sh->merge_abort = *abort;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (*reinterpret_cast<volatile int*>(&sh->merge_abort)) ok = false;
            if (ok) {
                tc_fence_after();
                // (m, l) of group 0 and group 1
                const float m0 = grp ? mo : (seen ? m_run : -INFINITY);
                const float l0 = grp ? lo : (seen ? l_run : -1.f);
                const float m1 = grp ? (seen ? m_run : -INFINITY) : mo;
                const float l1 = grp ? (seen ? l_run : -1.f) : lo;
                const bool has0 = l0 >= 0.f, has1 = l1 >= 0.f;
                const float m = fmaxf(m0, m1);
                uint32_t o0[32], o1[32];
                tmem_ld32(tmem + lane_off + COL_O + 32 * grp, o0);
                tmem_ld32(tmem + lane_off + COL_O + 64 + 32 * grp, o1);
                tmem_wait_ld();
                tc_fence_before();
                warp_arrive(&sh->o_free);
                if constexpr (!SPLIT) {
                    const float f0 = has0 ? ex2(m0 - m) : 0.f, f1 = has1 ? ex2(m1 - m) : 0.f;
                    const float lsum = (has0 ? l0 * f0 : 0.f) + (has1 ? l1 * f1 : 0.f);
                    const float inv = 1.f / lsum;
                    const float a0 = f0 * inv, a1 = f1 * inv;
                    // the row's log2-sum-exp of the scores (log2 units), kept
                    // for a backward pass
                    if (p.lse && grp == 0 && cur.i0 + ii < p.L &&
                        TXL_BOUNDS(cur.bh < p.B * p.H, 410, cur.bh))
                        p.lse[(size_t)cur.bh * p.L + cur.i0 + ii] = m + log2f(lsum);
                    // Each warp writes its 32 rows of the group's 32 output columns
                    // with one TMA store of a 32 x 32 box, staged in the upper
                    // 2 KB of the warp's own quarter of the P buffer (free: the
                    // group's last P V finished; the merge exchange uses the
                    // lower 1 KB of quarter 0) in the 64-byte swizzle the store
                    // expects: chunk c of row r at chunk c ^ ((r >> 1) & 3), which
                    // also spreads each 8-thread phase over all banks.  Only this
                    // warp writes its quarter again (scratch, P rows), after its
                    // lane 0 has seen the store read the box.
                    const uint32_t stage = p_tile + wq * 4096 + 2048;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float x0 = has0 ? __uint_as_float(o0[8 * c + e]) * a0 : 0.f;
                            y[e] = has1 ? fmaf(__uint_as_float(o1[8 * c + e]), a1, x0) : x0;
                        }
                        if (TXL_SMEM_IN(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), 16, 407))
                        st_shared_v4(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), pack_bf16x2(y[0], y[1]),
                                     pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && cur.i0 + 32 * wq < p.L) {
                        tma_store_3d(&tmO, stage, 32 * grp, cur.i0 + 32 * wq, cur.bh);
                        store_pending = true;
                    }
                } else {
                    // this unit's share: O relative to the row max m, and
                    // (m, l); a split unit may hold no visible key of a row
                    // (all its keys past the row's diagonal): zeros, l = 0
                    const bool live = m > -INFINITY;
                    const float f0 = (has0 && live) ? ex2(m0 - m) : 0.f;
                    const float f1 = (has1 && live) ? ex2(m1 - m) : 0.f;
                    float4* orow = reinterpret_cast<float4*>(
                        p.ws_o + ((size_t)cur.unit * BM + ii) * DH + 32 * grp);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float y[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x0 = has0 ? __uint_as_float(o0[4 * c + e]) * f0 : 0.f;
                            y[e] = has1 ? fmaf(__uint_as_float(o1[4 * c + e]), f1, x0) : x0;
                        }
                        if (TXL_BOUNDS(cur.unit < p.n_units, 408, cur.unit))
                            orow[c] = make_float4(y[0], y[1], y[2], y[3]);
                    }
                    if (grp == 0 && TXL_BOUNDS(cur.unit < p.n_units, 409, cur.unit))
                        p.ws_ml[(size_t)cur.unit * BM + ii] =
                            make_float2(m, (has0 ? l0 * f0 : 0.f) + (has1 ? l1 * f1 : 0.f));
                }
            }
            gbase += slots_of(cur.ntiles);
        }
        if (!SPLIT && lane == 0) bulk_wait_all();
        tc_fence_before();
    } else if (warp == 8) {
        // ------------------------------------------------ score MMA issuer
        // Key tiles go out in pairs (2p, 2p+1) of one item, one per softmax
        // group (group g takes the item's tiles t = g mod 2): one N=128 MMA
        // chain computes both tiles' AC into AC0|AC1 against the 128-key K box
        // of stage p, and one N=128 chain computes the two new position slots
        // 2p+2, 2p+3 (slots 0-3 for the first pair) against one R box.  The
        // pages' relative shift needs slots t, t+1, t+2 for tile t.
        //
        // Pair p overwrites both AC buffers and one slot pair (for p = 0 both)
        // whose earlier readers are tiles already issued, so it waits until
        // every issued tile has read its scores.  s_free of each group
        // completes once per tile of that group, in order, and cannot run two
        // phases ahead of these waits: its next phase needs the next pair.
        // The whole warp waits (bounded, voted); one elected lane issues.
        const uint32_t leader = elect_one();
        {
            bool ok = true;
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                if (ok)
                    ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kDevTimeoutMma, abort, p.status));
                return ok;
            };
            // Shared-memory descriptors of every operand buffer, precomputed;
            // a k-step of 16 elements (32 bytes) adds 2 to the address field
            // (16-byte units).
            const uint64_t dQ0 = smem_desc_sw128(s_base + OFF_Q, 16, 1024);
            const uint64_t dK0 = smem_desc_sw128(s_base + OFF_KV, 16, 1024);
            const uint64_t dR0 = smem_desc_sw128(s_base + OFF_R, 16, 1024);
            constexpr uint32_t U_Q = SZ_Q >> 4, U_BOX = SZ_BOX >> 4;
            int seen0 = 0, seen1 = 0;  // s_free completions observed, per group
            int iss0 = 0, iss1 = 0;    // tiles issued, per group
            int kv_s = 0, r_s = 0;     // K/V stage and R box counters at the item start
            int gbase = 0;             // global position-slot counter at the item start
            Item is;
            for (int ks = 0; ok && item_of<SPLIT, LOWER>(p, ks, is); ++ks) {
                const int npairs = (is.ntiles + 1) >> 1;
                const int nrb = npairs + 1;  // R boxes of the item (slots 0 .. 2*npairs+1)
                wait(&sh->q_ready, ks & 1);
                const uint64_t a_qu = dQ0 + (ks & 1) * 2 * U_Q;
                const uint64_t a_qv = a_qu + U_Q;
                int r_rel = 0;  // R boxes of this item released
                for (int pp = 0; ok && pp < npairs; ++pp) {
                    for (; ok && seen0 < iss0; ++seen0) wait(&sh->s_free[0], seen0 & 1);
                    for (; ok && seen1 < iss1; ++seen1) wait(&sh->s_free[1], seen1 & 1);
                    const int stage = kv_s + pp;
                    wait(&sh->kv_full[stage % KV_STAGES], (stage / KV_STAGES) & 1);
                    if (pp == 0) {
                        wait(&sh->r_full[r_s % R_STAGES], (r_s / R_STAGES) & 1);
                        wait(&sh->r_full[(r_s + 1) % R_STAGES], ((r_s + 1) / R_STAGES) & 1);
                    } else {
                        const int rb = r_s + pp + 1;
                        wait(&sh->r_full[rb % R_STAGES], (rb / R_STAGES) & 1);
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const bool two = 2 * pp + 1 < is.ntiles;
                    // AC of tiles 2p (AC0) and 2p+1 (AC1): the stage's K box
                    const uint64_t b_k = dK0 + (stage % KV_STAGES) * 2 * U_BOX;
                    const uint32_t idesc_ac = two ? IDESC_N128 : IDESC_N64;
#pragma unroll
                    for (int k = 0; k < DH / 16; ++k)
                        mma_ss_elect(tmem + COL_AC, a_qu + 2 * k, b_k + 2 * k, idesc_ac, k > 0, leader);
                    // position slots: R box b holds item slots 2b, 2b+1, which
                    // live in ring slot pair ((gbase / 2) + b) & 1
                    const int b_first = (pp == 0) ? 0 : pp + 1;
                    for (int b = b_first; b <= pp + 1; ++b) {
                        const uint64_t b_r = dR0 + ((r_s + b) % R_STAGES) * U_BOX;
                        const uint32_t d_r = tmem + COL_RING + 128 * (((gbase >> 1) + b) & 1);
#pragma unroll
                        for (int k = 0; k < DH / 16; ++k)
                            mma_ss_elect(d_r, a_qv + 2 * k, b_r + 2 * k, IDESC_N128, k > 0, leader);
                    }
                    if (leader) {
                        // the first pair of item ks: issued after q_ready of item
                        // ks and after every MMA of item ks-1
                        if (pp == 0) mma_commit(&sh->q_free);
                        if (!(p.inject == 1 && ks == 0 && pp == 0)) mma_commit(&sh->s_full[0]);
                        if (two) mma_commit(&sh->s_full[1]);
                        // R boxes 0 .. pp+1 are not read again
                        for (int b = r_rel; b <= pp + 1 && b < nrb; ++b)
                            mma_commit(&sh->r_empty[(r_s + b) % R_STAGES]);
                    }
                    r_rel = min(pp + 2, nrb);
                    ++iss0;
                    if (two) ++iss1;
                }
                kv_s += npairs;
                r_s += nrb;
                gbase += slots_of(is.ntiles);
            }
            if (leader) mma_commit(&sh->drain);
            drain_wait(&sh->drain, 0, p.status);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------------------------------------- P V MMA issuer
        // The tiles of each item in order; tile t belongs to group t mod 2.
        // PV(t) waits for the tile's P; the first P V of an item also for the
        // merge of the previous item to have read O.  p_full of a group cannot
        // complete twice before its P V is issued: the group's next P waits
        // for pv_done of this one.
        const uint32_t leader = elect_one();
        {
            bool ok = true;
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                if (ok)
                    ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kDevTimeoutMma, abort, p.status));
                return ok;
            };
            const uint64_t dP0 = smem_desc_sw128(s_base + OFF_P, 16, 1024);
            const uint64_t dV0 = smem_desc_sw128(s_base + OFF_KV + SZ_BOX, BN * 128, 1024);
            constexpr uint32_t U_Q = SZ_Q >> 4, U_T = SZ_T >> 4, U_BOX = SZ_BOX >> 4;
            Item ip;
            bool p_valid = item_of<SPLIT, LOWER>(p, 0, ip);
            int kp = 0, tp = 0, kv_p = 0;
            int pc0 = 0, pc1 = 0;  // P tiles consumed, per group
            while (ok && p_valid) {
                const int g = tp & 1;
                wait(&sh->p_full[g], (g ? pc1 : pc0) & 1);
                if (tp == 0 && kp > 0) wait(&sh->o_free, (kp - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                // K/V stage of tile tp; a stage is free once both of its tiles
                // went through P V (their S finished before their P existed)
                const int stage = kv_p + (tp >> 1);
                const uint64_t b_v = dV0 + (stage % KV_STAGES) * 2 * U_BOX + (tp & 1) * U_T;
                const uint64_t a_p = dP0 + g * U_Q;
                const uint32_t d_o = tmem + COL_O + 64 * g;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_ss_elect(d_o, a_p + 2 * k, b_v + 128 * k, IDESC_PV,
                                 (tp > 1 || k > 0) ? 1u : 0u, leader);
                if (leader) {
                    mma_commit(&sh->pv_done[g]);
                    if ((tp & 1) || tp == ip.ntiles - 1) mma_commit(&sh->kv_empty[stage % KV_STAGES]);
                    if (tp + 1 == ip.ntiles) mma_commit(&sh->o_done);
                }
                if (g) ++pc1; else ++pc0;
                if (++tp == ip.ntiles) {
                    kv_p += (ip.ntiles + 1) >> 1;
                    tp = 0;
                    ++kp;
                    p_valid = item_of<SPLIT, LOWER>(p, kp, ip);
                }
            }
            if (leader) mma_commit(&sh->drain);
            drain_wait(&sh->drain, 0, p.status);
        }
        __syncwarp();
    } else if (warp == 11) {
        // ------------------------------------------------ q+u, q+v operands
        // Item k's operands live in Q buffer k & 1: (q+u)c in slot 0, (q+v)c in
        // slot 1, c = scale * log2 e, rounded to bf16.  The raw q tile arrives
        // by TMA in both slots (128B swizzle: chunk ch of row r at chunk
        // ch ^ (r & 7); rows past L arrive as zeros) and is rewritten in place.
        // Item k >= 1 waits for q_free completion k-1 (the first pair of item
        // k-1 and everything before it completed): the issuer has consumed
        // q_ready of item k-1, so q_ready never runs two phases ahead of its
        // waits, and the score MMAs of item k-2, the last readers of buffer
        // k & 1, are done.  Likewise q_free completion k needs q_ready of item
        // k, so it never runs two phases ahead of this warp's waits.
        const float qscale = p.scale_log2;
        const int ch = lane & 7;  // the lane's 16-byte chunk of every row it converts
        bool ok = true;
        int issued = 1, landed = 1;  // q tiles loaded / observed (item 0: by the groups)
        Item it;
        for (int k = 1; ok && item_of<SPLIT, LOWER>(p, k, it); ++k) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&sh->q_free, (k - 1) & 1, kDevTimeoutMma, abort, p.status));
            if (!ok) break;
            const uint32_t qb = OFF_Q + (k & 1) * 2 * SZ_Q;
            if (lane == 0) {
                mbar_expect_tx(&sh->q_full, 2 * SZ_Q);
                tma_load_3d(smem + qb, &tmQ, &sh->q_full, 0, it.i0, it.bh);
                tma_load_3d(smem + qb + SZ_Q, &tmQ, &sh->q_full, 0, it.i0, it.bh);
            }
            ++issued;
            const bool hin = TXL_BOUNDS(it.h < p.H, 410, it.h);
            const uint4 bu = hin ? __ldg(reinterpret_cast<const uint4*>(p.ub + (size_t)it.h * DH) + ch)
                                 : make_uint4(0, 0, 0, 0);
            const uint4 bv = hin ? __ldg(reinterpret_cast<const uint4*>(p.vb + (size_t)it.h * DH) + ch)
                                 : make_uint4(0, 0, 0, 0);
            ok = __all_sync(0xffffffffu, mbar_wait(&sh->q_full, k & 1, kDevTimeoutMma, abort, p.status));
            if (!ok) break;
            ++landed;
#pragma unroll 4
            for (int r = lane >> 3; r < BM; r += 4) {
                const uint32_t a = s_base + qb + r * 128 + ((ch ^ (r & 7)) << 4);
#pragma unroll
                for (int slot = 0; slot < 2; ++slot) {
                    const uint4& b4 = slot ? bv : bu;
                    float raw[4];
                    if (!TXL_SMEM_IN(a + slot * SZ_Q, 16, 411)) continue;
                    ld_shared_v4(a + slot * SZ_Q, raw);
                    const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(raw);
                    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b4);
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 qf = __bfloat1622float2(q2[e]);
                        const float2 bf = __bfloat1622float2(b2[e]);
                        w[e] = pack_bf16x2((qf.x + bf.x) * qscale, (qf.y + bf.y) * qscale);
                    }
                    st_shared_v4(a + slot * SZ_Q, w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&sh->q_ready, 8);
        }
        // drain: a q tile still in flight lands before the CTA exits
        if (landed < issued) drain_wait(&sh->q_full, (issued - 1) & 1, p.status);
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------ TMA producers
        // Lane 0 streams the K/V stages (and warms L2 ahead of them), lane 1
        // the R boxes, each gated only by its own ring: a K/V stage still
        // held by P V does not hold back the next R box, nor the reverse.
        // The prologue ran on lane 0: every lane learns what it issued.
        pre_kv = __shfl_sync(0xffffffffu, pre_kv, 0);
        pre_r = __shfl_sync(0xffffffffu, pre_r, 0);
        if (lane == 0) {
            int kvc = pre_kv;  // K/V stages issued (item 0's first in the prologue)
            bool ok = true;
            Item it;
            for (int k = 0; ok && item_of<SPLIT, LOWER>(p, k, it); ++k) {
                const int nkv = (it.ntiles + 1) >> 1;  // K/V stages of this item
                for (int u = 0; u < nkv; ++u) {
                    if (k == 0 && u < pre_kv) {
                        // issued in the prologue; warm L2 for the next stages
                        for (int w = 1; w <= PREFETCH && w < nkv; ++w) {
                            tma_prefetch_l2_3d(&tmK, 0, (it.t0 + 2 * w) * BN, it.bh);
                            tma_prefetch_l2_3d(&tmV, 0, (it.t0 + 2 * w) * BN, it.bh);
                            tma_prefetch_l2_2d(&tmR, it.h * DH, it.rbase + SLOT * 2 * (w + 1));
                        }
                        continue;
                    }
                    const int s = kvc % KV_STAGES;
                    if (kvc >= KV_STAGES && !mbar_wait(&sh->kv_empty[s], ((kvc / KV_STAGES) & 1) ^ 1,
                                                       kDevTimeoutProducer, abort, p.status)) {
                        ok = false;
                        break;
                    }
                    // warm L2 PREFETCH stages ahead (the first ones at the item start)
                    for (int w = (u == 0 ? 1 : u + PREFETCH); w <= u + PREFETCH && w < nkv; ++w) {
                        tma_prefetch_l2_3d(&tmK, 0, (it.t0 + 2 * w) * BN, it.bh);
                        tma_prefetch_l2_3d(&tmV, 0, (it.t0 + 2 * w) * BN, it.bh);
                        tma_prefetch_l2_2d(&tmR, it.h * DH, it.rbase + SLOT * 2 * (w + 1));
                    }
                    mbar_expect_tx(&sh->kv_full[s], 2 * SZ_BOX);
                    uint8_t* st = smem + OFF_KV + s * 2 * SZ_BOX;
                    tma_load_3d(st, &tmK, &sh->kv_full[s], 0, (it.t0 + 2 * u) * BN, it.bh);
                    tma_load_3d(st + SZ_BOX, &tmV, &sh->kv_full[s], 0, (it.t0 + 2 * u) * BN, it.bh);
                    ++kvc;
                }
            }
            // drain: the last load into each ring slot has landed
            for (int c = kvc - KV_STAGES; c < kvc; ++c)
                if (c >= 0) drain_wait(&sh->kv_full[c % KV_STAGES], (c / KV_STAGES) & 1, p.status);
        } else if (lane == 1) {
            int rc = pre_r;  // R boxes issued (item 0's first in the prologue)
            bool ok = true;
            Item it;
            for (int k = 0; ok && item_of<SPLIT, LOWER>(p, k, it); ++k) {
                const int nrb = (it.ntiles + 3) >> 1;  // R boxes: slots 0 .. ntiles+1
                for (int rb = (k == 0 ? pre_r : 0); rb < nrb; ++rb, ++rc) {
                    const int s = rc % R_STAGES;
                    if (rc >= R_STAGES && !mbar_wait(&sh->r_empty[s], ((rc / R_STAGES) & 1) ^ 1,
                                                     kDevTimeoutProducer, abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&sh->r_full[s], SZ_BOX);
                    tma_load_2d(smem + OFF_R + s * SZ_BOX, &tmR, &sh->r_full[s], it.h * DH,
                                it.rbase + SLOT * 2 * rb);
                }
            }
            for (int c = rc - R_STAGES; c < rc; ++c)
                if (c >= 0) drain_wait(&sh->r_full[c % R_STAGES], (c / R_STAGES) & 1, p.status);
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

// Combines the key splits of every query row: with m* the largest split max
// of the row, out = sum_s 2^(m_s - m*) O_s / sum_s 2^(m_s - m*) l_s (the
// online-softmax merge of partial results).  One thread per 8 output columns.
__global__ void __launch_bounds__(256)
attn_combine_kernel(const float* __restrict__ ws_o, const float2* __restrict__ ws_ml,
                    __nv_bfloat16* __restrict__ out, int n_bh, int L, int n_qtiles, int nsplit) {
    using namespace tc;
    const int t = blockIdx.x * 256 + threadIdx.x;
    if (t >= n_bh * L * 8) return;
    const int ch = t & 7, row = t >> 3;
    const int i = row % L, bh = row / L;
    const int qt = i / BM, ii = i % BM;
    const int witem = (n_qtiles - 1 - qt) * n_bh + bh;
    // every unit this row reads exists: n_bh * n_qtiles items of nsplit units
    if (!TXL_BOUNDS((long long)(witem + 1) * nsplit <= (long long)n_bh * n_qtiles * nsplit, 412, witem)) return;
    float mx = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) {
        const float2 ml = ws_ml[(size_t)(witem * nsplit + sp) * BM + ii];
        if (ml.y > 0.f) mx = fmaxf(mx, ml.x);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, den = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
        const size_t unit = (size_t)witem * nsplit + sp;
        const float2 ml = ws_ml[unit * BM + ii];
        if (!(ml.y > 0.f)) continue;
        const float w = exp2f(ml.x - mx);
        den += w * ml.y;
        const float4* o = reinterpret_cast<const float4*>(ws_o + (unit * BM + ii) * DH + 8 * ch);
        const float4 a = o[0], b = o[1];
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
        acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
    const float inv = 1.f / den;
    uint4 r;
    r.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    r.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    r.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    r.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    reinterpret_cast<uint4*>(out + ((size_t)bh * L + i) * DH)[ch] = r;
}

// ---------------------------------------------------------------- host side
static int num_sms() { return current_sm_count(); }

// Launch with programmatic stream serialisation (the kernel waits for the
// previous kernel of the stream before its first global access).
template <typename Kern>
static void launch_pdl(Kern kern, int grid, cudaStream_t stream, const CUtensorMap& a, const CUtensorMap& b,
                       const CUtensorMap& c, const CUtensorMap& d, const CUtensorMap& e, const TcParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc::NTHREADS);
    cfg.dynamicSmemBytes = tc::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kern, a, b, c, d, e, p);
}

// Returns cudaErrorInvalidValue if a tensor map cannot be encoded.
// Key splits per item when a workspace is available.  With fewer items than
// SMs, whole items leave SMs idle; splitting each item's key tiles over
// several units fills them, at the price of per-unit work (the q tile, the
// first pair's extra position slots, the partial result) and a combine pass.
// The count minimises a makespan estimate in key tiles: rounds of units per
// CTA times (tiles per unit + kUnitCost), plus kCombineCost when split.
// Every split keeps at least two tile pairs.
int attn_tc_bf16_splits(int B, int H, int L, int M) {
    using namespace tc;
    constexpr double kUnitCost = 3.0, kCombineCost = 4.0;  // in key tiles, measured on GB300
    const long long n_items = (long long)B * H * ((L + BM - 1) / BM);
    const int sms = num_sms();
    if (n_items >= sms || n_items <= 0) return 1;
    const int tiles_max = (M + L - 1) / BN + 1;                 // longest item
    const int tiles0 = (M + (L < BM ? L : BM) - 1) / BN + 1;   // shortest item
    const int max_split = ((tiles0 + 1) / 2) / 2;
    int best = 1;
    double best_cost = 1e300;
    for (int ns = 1; ns <= max_split || ns == 1; ++ns) {
        const long long units = n_items * ns;
        const double rounds = (double)((units + sms - 1) / sms);
        const double cost = rounds * ((double)tiles_max / ns + kUnitCost) + (ns > 1 ? kCombineCost : 0.0);
        if (cost < best_cost) {
            best_cost = cost;
            best = ns;
        }
        if (ns >= 64) break;
    }
    return best;
}

// Workspace bytes of a split launch (0 when the launch does not split):
// per unit, O [128][64] and (m, l) [128] in fp32.
size_t attn_tc_bf16_workspace_bytes(int B, int H, int L, int M) {
    using namespace tc;
    const int ns = attn_tc_bf16_splits(B, H, L, M);
    if (ns <= 1) return 0;
    const size_t units = (size_t)B * H * ((L + BM - 1) / BM) * ns;
    return units * BM * (DH * sizeof(float) + sizeof(float2));
}

// The launch behind both entry points below.
static cudaError_t launch_tc(const void* q, const void* k, const void* v, const void* r, const void* ub,
                             const void* vb, int B, int H, int L, int M, float scale, int lo_shift, void* out,
                             void* workspace, float* lse, int inject, int* status, cudaStream_t stream) {
    using namespace tc;
    static PerDeviceOnce attrs;
    {
        const cudaError_t e = attrs.run([] {
            cudaError_t r = cudaFuncSetAttribute(attn_tc_bf16_kernel<false, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(attn_tc_bf16_kernel<true, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(attn_tc_bf16_kernel<false, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            return r;
        });
        if (e != cudaSuccess) return e;
    }
    const int K = M + L;
    CUtensorMap mQ, mK, mV, mR, mO;
    {
        // q tile of an item: 128 rows of one (b, h); rows past L read as zeros
        cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)L, (cuuint64_t)B * H};
        cuuint64_t strides[2] = {(cuuint64_t)DH * 2, (cuuint64_t)L * DH * 2};
        cuuint32_t box[3] = {DH, BM, 1};
        if (!encode_bf16(&mQ, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
        // output: one warp's 32 rows x one group's 32 columns per store (rows
        // past L clipped)
        cuuint32_t obox[3] = {DH / 2, 32, 1};
        if (!encode_bf16(&mO, out, 3, dims, strides, obox, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)K, (cuuint64_t)B * H};
        cuuint64_t strides[2] = {(cuuint64_t)DH * 2, (cuuint64_t)K * DH * 2};
        cuuint32_t box[3] = {DH, 2 * BN, 1};
        if (!encode_bf16(&mK, k, 3, dims, strides, box)) return cudaErrorInvalidValue;
        if (!encode_bf16(&mV, v, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)H * DH, (cuuint64_t)K};
        cuuint64_t strides[1] = {(cuuint64_t)H * DH * 2};
        cuuint32_t box[2] = {DH, 2 * SLOT};
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
    p.lo_shift = lo_shift;
    p.n_qtiles = (L + BM - 1) / BM;
    const long long n_items = (long long)B * H * p.n_qtiles;
    if (n_items > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    p.n_items = (int)n_items;
    // the same_length bound runs unsplit (txl_attn_fwd_ex takes no workspace)
    const bool lower = lo_shift < (1 << 30);
    p.nsplit = (workspace && !lower) ? attn_tc_bf16_splits(B, H, L, M) : 1;
    if ((long long)p.n_items * p.nsplit + 2ll * num_sms() >= 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    p.n_units = p.n_items * p.nsplit;
    const size_t units = (size_t)p.n_units;
    p.ws_o = p.nsplit > 1 ? static_cast<float*>(workspace) : nullptr;
    p.ws_ml = p.nsplit > 1 ? reinterpret_cast<float2*>(static_cast<float*>(workspace) + units * BM * DH)
                           : nullptr;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse = lse;
    if (lse && p.nsplit > 1) return cudaErrorInvalidValue;  // the unsplit kernel writes it
    p.inject = inject;
    p.status = status;
    const int grid = p.n_units < num_sms() ? p.n_units : num_sms();
    if (p.nsplit > 1)
        launch_pdl(attn_tc_bf16_kernel<true, false>, grid, stream, mQ, mK, mV, mR, mO, p);
    else if (lower)
        launch_pdl(attn_tc_bf16_kernel<false, true>, grid, stream, mQ, mK, mV, mR, mO, p);
    else
        launch_pdl(attn_tc_bf16_kernel<false, false>, grid, stream, mQ, mK, mV, mR, mO, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.nsplit == 1) return e;
    const long long threads = (long long)B * H * L * 8;
    if (threads >= 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    attn_combine_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(
        p.ws_o, p.ws_ml, p.out, B * H, L, p.n_qtiles, p.nsplit);
    return cudaGetLastError();
}

cudaError_t launch_attn_tc_bf16(const void* q, const void* k, const void* v, const void* r,
                                const void* ub, const void* vb, int B, int H, int L, int M,
                                float scale, int lo_shift, void* out, void* workspace, int inject,
                                int* status, cudaStream_t stream) {
    return launch_tc(q, k, v, r, ub, vb, B, H, L, M, scale, lo_shift, out, workspace, nullptr, inject, status,
                     stream);
}

// The unsplit forward that also leaves each row's log2-sum-exp of the scores
// in lse [B*H][L] (fp32, log2 units: P = 2^(scale log2 e (AC+BD) - lse)).
cudaError_t launch_attn_tc_bf16_lse(const void* q, const void* k, const void* v, const void* r, const void* ub,
                                    const void* vb, int B, int H, int L, int M, float scale, int lo_shift,
                                    void* out, float* lse, int* status, cudaStream_t stream) {
    if (!lse) return cudaErrorInvalidValue;
    return launch_tc(q, k, v, r, ub, vb, B, H, L, M, scale, lo_shift, out, nullptr, lse, 0, status, stream);
}

TXL_BOUNDS_READER(bounds_word_attn_tc)

}  // namespace txl
