// Backward pass of the fused Transformer-XL relative attention on the
// sm_103a tensor cores (tcgen05 + TMEM, TMA-staged operands): bf16 inputs,
// d_h = 64, fp32 gradients of sum(out * dout).
//
// With s_ij = scale ((q_i+u).k_j + (q_i+v).R_{r(i,j)}) on the visible pairs
// (key j <= M + i; R row r(i,j) = L-1-i+j holds distance M+i-j), P = softmax_j
// s, out_i = sum_j P_ij v_j ("Transformer-XL模型 核心源码阅读笔记", section
// "Build the model", RelPartialLearnableMultiHeadAttn.forward; the memory is
// a constant input of the segment, the "Transformer-XL" notes, section
// "Segment-Level Recurrence"):
//
//   dv_j  = sum_i P_ij dout_i
//   dP_ij = dout_i . v_j,  D_i = dout_i . out_i,  dS_ij = P_ij (dP_ij - D_i)
//   dq_i  = scale sum_j dS_ij (k_j + R_{r(i,j)})
//   dk_j  = scale sum_i dS_ij (q_i + u)
//   dR_r  = scale sum over b and the pairs (i, j) with r(i,j) = r of dS_ij (q_i + v)
//   du    = scale sum dS_ij k_j,   dv_bias = scale sum dS_ij R_{r(i,j)}
//
// Passes, in order on one stream:
//   1. the forward kernel writing the output and each query row's log2-sum-
//      exp lse into the workspace (launch_attn_tc_bf16_lse); skipped when the
//      caller passes the forward's saved output and lse
//   2. attn_bwd_prep_kernel: per query row D = dout . out, and the score
//      operands (q+u)c, (q+v)c as bf16 (c = scale log2 e), rounded exactly as
//      the forward rounds them
//   3. attn_bwd_q_kernel, query-major like the forward: one item is a
//      (b, h, 128-row query tile) and all its key tiles of 64.  It recomputes
//      the scores (content AC plus the position band read through the same
//      per-row shift as the forward), P = 2^(s - lse), dP = dout V^T, dS, and
//      accumulates in TMEM dq_c = dS K and dq_p = G R, where G is dS moved to
//      band coordinates (row ii's key jj of tile t at band column
//      64 t + 127 - ii + jj, the relative shift run backwards).  Every
//      completed pair of 64-column band slots also gives dR = G^T (q+v)
//      (an MMA with G read transposed), which four flush warps add to the
//      fp32 dR with vector reductions.  du and dv_bias are the row sums of
//      dq_c and dq_p.
//   4. attn_bwd_kv_kernel, key-major: one item is a (b, h, 128-key tile) and
//      every 128-row query tile that sees it.  It recomputes the scores of
//      the 128 x 128 block (the position band as one N = 256 MMA), P, dP and
//      dS, and accumulates in TMEM dV = P^T dout and dK = dS^T (q+u) (P and
//      dS read transposed from the buffer the threads write them to).
//
// The 1 / log2 e of the gradients taken through (q+u)c and (q+v)c (dK, dR)
// and the scale of dq are applied when the accumulators are read.  Every
// mbarrier wait is bounded (1 s of %globaltimer); on expiry the CTA records a
// status, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_tc_common.cuh"
#include "txl_device.cuh"

namespace txl {

namespace bw {
constexpr int BM = 128;  // query rows per tile (TMEM lanes)
constexpr int BN = 64;   // keys per tile of the query-major pass
constexpr int DH = 64;   // head dim: one 128-byte swizzle row
constexpr uint32_t SZ_T = BN * DH * 2;  //  8 KB: 64 rows of d_h
constexpr uint32_t SZ_Q = BM * DH * 2;  // 16 KB: 128 rows of d_h (or 128 x 64 bf16)
constexpr float kLn2 = 0.69314718055994531f;

// ---- attn_bwd_q_kernel (query-major)
// warps 0-3 softmax (one query row per thread), 4 score issuer (AC, the
// position slots, dP), 5 TMA producer of the q-side tiles and K/V, 6-9 band
// scatter / dR / dq (row quarter w%4), 10 gradient issuer (dq_c, dq_p, dR),
// 11 TMA producer of the R boxes
constexpr int QA_THREADS = 384;
constexpr int QA_KV = 2;     // K/V ring, one 64-key tile per stage
constexpr int QA_RB = 3;     // R ring, one 128-row box (two band slots) per stage
constexpr int QA_G = 4;      // G ring (band slots of dS) in shared memory
constexpr int QA_RING = 3;   // position slots in TMEM: tile t reads slots t, t+1, t+2
constexpr uint32_t QA_OFF_QU = 0;
constexpr uint32_t QA_OFF_DO = QA_OFF_QU + SZ_Q;
constexpr uint32_t QA_OFF_QV = QA_OFF_DO + SZ_Q;
constexpr uint32_t QA_OFF_KV = QA_OFF_QV + SZ_Q;          // stage s: K at +16K*s, V at +16K*s+8K
constexpr uint32_t QA_OFF_R = QA_OFF_KV + QA_KV * 2 * SZ_T;
constexpr uint32_t QA_OFF_DS = QA_OFF_R + QA_RB * SZ_Q;   // dS tiles (tile parity); each also the shift scratch
constexpr uint32_t QA_OFF_G = QA_OFF_DS + 2 * SZ_Q;       // G slot g at +16K*g
constexpr uint32_t QA_OFF_BAR = QA_OFF_G + QA_G * SZ_Q;
constexpr uint32_t QA_SMEM = QA_OFF_BAR + 1024 + 1024;
static_assert(QA_SMEM <= 232448, "shared memory budget of one sm_103a CTA");
// TMEM columns: AC 0-63, dP 64-127, position ring 128-319, dR 320-383, dq_c, dq_p
constexpr uint32_t QA_COL_S = 0, QA_COL_DP = 64, QA_COL_RING = 128, QA_COL_DR = 320, QA_COL_DQC = 384,
                   QA_COL_DQP = 448;

// ---- attn_bwd_kv_kernel (key-major)
// warps 0-7 softmax (two threads per query row: warp w takes keys 64 (w/4)
// .. of the block, rows of lane quarter w%4), 8 MMA issuer, 9 TMA producer of
// K/V and the q-side stages, 10 TMA producer of (q+v)c and the R band (a warp
// of its own: two lanes of one warp in blocking waits hold each other up)
constexpr int KB_THREADS = 352;
constexpr uint32_t KB_OFF_KV = 0;                       // buffer b: K at +32K*b, V at +32K*b+16K
constexpr uint32_t KB_OFF_ST = KB_OFF_KV + 4 * SZ_Q;    // stage s: (q+u)c at +32K*s, dout at +32K*s+16K
constexpr uint32_t KB_OFF_QV = KB_OFF_ST + 4 * SZ_Q;
constexpr uint32_t KB_OFF_R = KB_OFF_QV + SZ_Q;         // 256 R rows
constexpr uint32_t KB_OFF_P = KB_OFF_R + 2 * SZ_Q;      // P then dS: key half h at +16K*h
constexpr uint32_t KB_OFF_BAR = KB_OFF_P + 2 * SZ_Q;
constexpr uint32_t KB_SMEM = KB_OFF_BAR + 1024 + 1024;
static_assert(KB_SMEM <= 232448, "shared memory budget of one sm_103a CTA");
// TMEM columns: AC then dP 0-127, position band 128-383, dK, dV
constexpr uint32_t KB_COL_S = 0, KB_COL_BAND = 128, KB_COL_DK = 384, KB_COL_DV = 448;

constexpr uint32_t IDESC_N64 = idesc_bf16_f32(128, 64, 0);          // B K-major, 64 rows
constexpr uint32_t IDESC_N128 = idesc_bf16_f32(128, 128, 0);        // B K-major, 128 rows
constexpr uint32_t IDESC_N256 = idesc_bf16_f32(128, 256, 0);        // B K-major, 256 rows
constexpr uint32_t IDESC_N64_BMN = idesc_bf16_f32(128, 64, 1);      // B MN-major (d_h contiguous)
constexpr uint32_t IDESC_N64_ABMN = idesc_bf16_f32(128, 64, 1, 1);  // A and B MN-major
}  // namespace bw

struct BwdParams {
    int B, H, L, M, K;     // K = M + L keys
    int n_qtiles;          // 128-row query tiles
    int n_ktiles;          // 128-key tiles (key-major pass)
    int n_items;
    const float2* stats;   // [B*H][L]: (lse in log2 units, D)
    float* dq;             // [B*H][L][64]
    float* dk;             // [B*H][K][64]
    float* dv;             // [B*H][K][64]
    float* dr;             // [K][H][64], accumulated
    float* du;             // [H][64], accumulated
    float* dvb;            // [H][64], accumulated
    float scale;
    int* status;
};

struct QaShared {
    uint64_t kv_full[bw::QA_KV], kv_empty[bw::QA_KV];
    uint64_t r_full[bw::QA_RB], r_empty[bw::QA_RB];
    uint64_t qa_full, qa_empty;    // (q+u)c and dout of the item landed / no longer read
    uint64_t qv_full, qv_empty;    // (q+v)c of the item
    uint64_t s_full, s_free;     // AC and the tile's band slots are in TMEM / have been read
    uint64_t dp_full, dp_free;   // dP of the tile is in TMEM / has been read
    uint64_t ds_full[2];         // dS tile b (tile parity) is in shared memory
    uint64_t ds_read[2];         // the flush warps have read dS tile b
    uint64_t dqc_done[2];        // the dq_c MMA that reads dS tile b completed
    uint64_t g_full;             // the tile's band scatter is in G
    uint64_t post;               // the MMAs after the scatter (and all before) completed
    uint64_t dr_full, dr_free;   // a dR pair is in TMEM / the flush warps read it
    uint64_t dq_done;            // every MMA of the item completed
    uint64_t dq_free;            // the flush warps read the item's dq accumulators
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort;
};

struct KbShared {
    uint64_t kv_full[2], kv_empty[2];
    uint64_t q_full[2], q_empty[2];  // (q+u)c and dout of a step
    uint64_t qv_full, qv_empty;      // (q+v)c of a step
    uint64_t r_full, r_empty;        // the R band of a step
    uint64_t s_full, s_free;
    uint64_t dp_full, dp_free;
    uint64_t pt_full, pv_done;       // P in shared memory / dV MMA done with it
    uint64_t ds_full, post;          // dS in shared memory / dK MMA done with it
    uint64_t dkv_done;               // every MMA of the item completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Query-major item k of this CTA: (b, h, query tile), longest query tile
// first, dealt to CTAs in snake order (the forward's order).
struct QaItem {
    int bh, h, i0, nt, rbase;
};
__device__ __forceinline__ bool qa_item(const BwdParams& p, int k, QaItem& it) {
    const int G = gridDim.x, c = blockIdx.x;
    const int w = k * G + ((k & 1) ? (G - 1 - c) : c);
    if (w >= p.n_items) return false;
    const int n_bh = p.B * p.H;
    const int qq = w / n_bh;
    const int qt = p.n_qtiles - 1 - qq;
    it.bh = w - qq * n_bh;
    it.h = it.bh % p.H;
    it.i0 = qt * bw::BM;
    const int rows = min(bw::BM, p.L - it.i0);
    it.nt = (p.M + it.i0 + rows - 1) / bw::BN + 1;
    it.rbase = p.L - it.i0 - bw::BM;  // R row of band slot 0
    return true;
}
// Band slots an item occupies in the rings (0 .. nt+1, rounded up to even).
__device__ __forceinline__ int qa_slots(int nt) { return 2 * (((nt + 1) >> 1) + 1); }

// Key-major item k: (b, h, 128-key tile), lowest key tile (most query tiles)
// first.  Query tiles qlo .. n_qtiles-1 see some key of the tile.
struct KbItem {
    int bh, h, j0, qlo, nsteps;
};
__device__ __forceinline__ bool kb_item(const BwdParams& p, int k, KbItem& it) {
    const int G = gridDim.x, c = blockIdx.x;
    const int w = k * G + ((k & 1) ? (G - 1 - c) : c);
    if (w >= p.n_items) return false;
    const int n_bh = p.B * p.H;
    const int kt = w / n_bh;
    it.bh = w - kt * n_bh;
    it.h = it.bh % p.H;
    it.j0 = kt * 128;
    // row i sees key j iff i >= j - M: the tile's first key j0 is seen from
    // row j0 - M on
    const int first_row = it.j0 - p.M;
    it.qlo = first_row > 0 ? first_row / bw::BM : 0;
    it.nsteps = p.n_qtiles - it.qlo;
    return true;
}

// Warp-wide sum of 32 values per lane: lane l ends with the sum over the
// warp of column l (a butterfly reduce-scatter, 31 shuffles).
__device__ __forceinline__ float warp_sum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
    // level l: each lane holds 32 >> l partial columns; the lanes with bit
    // (16 >> l) set keep the upper half of them, their partners the lower
#pragma unroll
    for (int l = 0; l < 5; ++l) {
        const int bit = 16 >> l, hl = 16 >> l;
        const bool up = (lane & bit) != 0;
#pragma unroll
        for (int x = 0; x < hl; ++x) {
            const float send = up ? v[x] : v[x + hl];
            const float keep = up ? v[x + hl] : v[x];
            v[x] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    return v[0];
}

// bf16 halves: (hi of a, lo of b) when odd, else a
__device__ __forceinline__ uint32_t prmt_sel(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ void ld_shared_v4u(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr) : "memory");
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// One 16-byte chunk of the G ring: item band column 8 * ch .. 8 * ch + 7 of
// row ii (slot ch / 8, ring position (gslot + slot) % 4, 128-byte swizzle).
__device__ __forceinline__ uint32_t g_chunk_addr(uint32_t g_base, int gslot, int ch, int ii) {
    const int pos = (gslot + (ch >> 3)) & (bw::QA_G - 1);
    return g_base + pos * bw::SZ_Q + (ii >> 3) * 1024 + (ii & 7) * 128 + ((((ch & 7) ^ (ii & 7))) << 4);
}

// Scatter of one dS row of a key tile into band coordinates.  Row ii's key jj
// of tile t lands on item band column 64 t + o + jj (o = 127 - ii).  The
// chunk grid of 8 columns starts e = o % 8 columns before the row's first
// value: the chunk holding column 64 t + o - e .. carries the previous
// tile's last e values (cw, words 28-31 of its row), so every chunk is
// written whole, exactly once per item.  w[0..31]: this tile's values as
// bf16 pairs (2m, 2m+1).
// Output word x of the tile (columns C + 2x, C + 2x + 1, C = 64 t + o - e) is
// the stream element pair (s0 + 2x, s0 + 2x + 1), s0 = 8 - e, of
// S = [cw | w] (72 values): a half-word shift when s0 is odd (prmt), then a
// word shift by a' in 0..4 (three select stages).
__device__ __forceinline__ void g_align(const uint32_t (&cw)[4], const uint32_t (&w)[32], int e,
                                        uint32_t (&out)[32]) {
    const int s0 = 8 - e;
    const uint32_t sel = (s0 & 1) ? 0x5432u : 0x3210u;
    const int a = (s0 & 1) ? (s0 - 1) >> 1 : s0 >> 1;
    uint32_t v[40];
#pragma unroll
    for (int x = 0; x < 36; ++x) {
        const uint32_t lo = x < 4 ? cw[x] : w[x - 4];
        const uint32_t hi = x + 1 < 4 ? cw[x + 1] : (x + 1 < 36 ? w[x - 3] : 0u);
        v[x] = prmt_sel(lo, hi, sel);
    }
#pragma unroll
    for (int x = 36; x < 40; ++x) v[x] = 0u;
#pragma unroll
    for (int x = 0; x < 39; ++x) v[x] = (a & 1) ? v[x + 1] : v[x];
#pragma unroll
    for (int x = 0; x < 37; ++x) v[x] = (a & 2) ? v[x + 2] : v[x];
#pragma unroll
    for (int x = 0; x < 32; ++x) out[x] = (a & 4) ? v[x + 4] : v[x];
}

#define QA_SMEM_IN(addr, bytes, site) \
    TXL_BOUNDS((addr) >= s_base && (addr) + (bytes) <= s_base + bw::QA_SMEM, (site), (long long)(addr) - s_base)
#define KB_SMEM_IN(addr, bytes, site) \
    TXL_BOUNDS((addr) >= s_base && (addr) + (bytes) <= s_base + bw::KB_SMEM, (site), (long long)(addr) - s_base)

// --------------------------------------------------------------------------
// attn_bwd_q_kernel: dq, dR, du, dv_bias.
//
// Per key tile t of an item (global tile counter gt across items):
//   score issuer (warp 4):  AC(t) = (q+u)c K_t^T -> S and the position MMA of
//            band slot t+2 (slots 0-2 for t = 0) into a 3-slot TMEM ring
//            (the forward's rolling band, one slot per tile), then
//            dP(t) = dout V_t^T -> DP
//   softmax (warps 0-3, one query row per thread): reads AC and the tile's
//            band (releases them), shifts the band, P = 2^(s - lse), reads
//            dP (releases it), dS = P (dP - D) -> the dS tile (K-major)
//   flush (warps 6-9, row 32 (w%4) + lane): reads its row of the dS tile,
//            scatters it into G (band coordinates), reads and reduces each
//            dR pair into dr, and after the item's last tile writes dq and
//            adds the row sums of dq_c, dq_p to du, dv_bias
//   gradient issuer (warp 10): dq_c += dS K_t once the dS tile is in shared
//            memory; once the tile's scatter is in G, dq_p += G_slot R_slot
//            for the band slots complete after tile t (slot t; after the
//            last tile also nt, nt+1) and dR = G^T (q+v)c of each complete
//            slot pair -> DR
// The two issuers run independent chains: the scores and dP of the next
// tile go out as soon as the softmax has read the current ones.  G slot g is
// complete once tile g has been scattered (tile t writes slots t, t+1, t+2);
// a slot's position in the 4-slot G ring is rewritten two tiles later,
// after the flush warps have waited for `post` of the tile before.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(bw::QA_THREADS, 1)
attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tmQu, const __grid_constant__ CUtensorMap tmQv,
                  const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmR,
                  const BwdParams p) {
    using namespace bw;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    QaShared* sh = reinterpret_cast<QaShared*>(smem + QA_OFF_BAR);
    const uint32_t s_base = smem_u32(smem);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (warp == 4) {
        tmem_alloc(&sh->tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 5 && lane == 0) {
        tma_prefetch_desc(&tmQu);
        tma_prefetch_desc(&tmQv);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmR);
        // buffers read by both issuers are released by a commit of each
        for (int s = 0; s < QA_KV; ++s) {
            mbar_init(&sh->kv_full[s], 1);
            mbar_init(&sh->kv_empty[s], 2);
        }
        for (int s = 0; s < QA_RB; ++s) {
            mbar_init(&sh->r_full[s], 1);
            mbar_init(&sh->r_empty[s], 2);
        }
        mbar_init(&sh->qa_full, 1);
        mbar_init(&sh->qa_empty, 1);
        mbar_init(&sh->qv_full, 1);
        mbar_init(&sh->qv_empty, 2);
        mbar_init(&sh->s_full, 1);
        mbar_init(&sh->s_free, 4);
        mbar_init(&sh->dp_full, 1);
        mbar_init(&sh->dp_free, 4);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh->ds_full[b], 4);
            mbar_init(&sh->ds_read[b], 4);
            mbar_init(&sh->dqc_done[b], 1);
        }
        mbar_init(&sh->g_full, 4);
        mbar_init(&sh->post, 1);
        mbar_init(&sh->dr_full, 1);
        mbar_init(&sh->dr_free, 4);
        mbar_init(&sh->dq_done, 1);
        mbar_init(&sh->dq_free, 4);
        mbar_init(&sh->drain[0], 1);
        mbar_init(&sh->drain[1], 1);
        sh->abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The prep kernel's outputs (and the zeroed dR, du, dv_bias) are
    // complete: this grid starts after it.  The key-major pass, which reads
    // none of this kernel's outputs, may be scheduled on the SMs it leaves.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;
    const uint32_t ds_tile = s_base + QA_OFF_DS;

    if (warp < 4) {
        // ---------------------------------------------------------- softmax
        const int wq = warp;
        const int ii = tid;                      // query row within the item
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        // the warp's quarter of the tile's dS buffer doubles as its shift
        // scratch (written by this tile, read by tile t-2's MMA and flush)
        const uint32_t t_ld0 = ds_tile + wq * 4096 + 4 * lane;
        bool ok = true;
        int gt = 0, gring = 0;  // global tile, global position slot of the item's slot 0
        QaItem it;
        for (int k = 0; ok && qa_item(p, k, it); ++k) {
            const int i = it.i0 + ii;
            float lse = INFINITY, Dv = 0.f;  // rows past L: P = 0
            if (i < p.L) {
                const float2 st = p.stats[(size_t)it.bh * p.L + i];
                lse = st.x;
                Dv = st.y;
            }
            for (int t = 0; t < it.nt; ++t, ++gt) {
                const int db = gt & 1;  // dS buffer of the tile
                const uint32_t t_ld = t_ld0 + db * SZ_Q;
                const uint32_t t_st = t_ld - 128u * (uint32_t)(31 - lane);
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->s_full, gt & 1, kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
                tc_fence_after();
                float sc[64];
                {
                    // the band first (packed and stored to the shift scratch),
                    // then AC: the two are never held in registers together
                    uint32_t hp[64];
                    {
                        uint32_t bwv[96];
#pragma unroll
                        for (int kc = 0; kc < 3; ++kc) {
                            const int c = 96 - 32 * wq + 32 * kc;
                            const uint32_t rc = QA_COL_RING + 64 * ((gring + t + (c >> 6)) % QA_RING) + (c & 63);
                            tmem_ld32(tmem + lane_off + rc, *reinterpret_cast<uint32_t(*)[32]>(&bwv[32 * kc]));
                        }
                        tmem_wait_ld();
#pragma unroll
                        for (int K = 0; K < 64; ++K)
                            hp[K] = pack_f16x2_sat(__uint_as_float(bwv[K]), __uint_as_float(bwv[K + 32]));
                    }
                    // the scratch (this tile's dS buffer) is free once tile
                    // gt-2's dq_c MMA and the flush warps have read it
                    if (gt >= 2) {
                        const uint32_t ph = ((gt - 2) >> 1) & 1;
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait(&sh->dqc_done[db], ph, kDevTimeoutSoftmax, abort, p.status) &&
                                            mbar_wait(&sh->ds_read[db], ph, kDevTimeoutSoftmax, abort, p.status));
                    }
                    if (!ok) break;
                    __syncwarp();
                    if (!QA_SMEM_IN(t_ld, 128 * 31 + 4, 701)) break;
                    st_shift_all<0>(31 - lane, t_st, *reinterpret_cast<uint32_t(*)[32]>(&hp[0]),
                                    *reinterpret_cast<uint32_t(*)[32]>(&hp[32]));
                    uint32_t ac[64];
                    tmem_ld32(tmem + lane_off + QA_COL_S, *reinterpret_cast<uint32_t(*)[32]>(&ac[0]));
                    tmem_ld32(tmem + lane_off + QA_COL_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&ac[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    warp_arrive(&sh->s_free);
                    float win[32];
                    ld_shift_all<0>(t_ld, win);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const float2 s2 = add_h2_f32(__float_as_uint(win[x]), __uint_as_float(ac[x]),
                                                     __uint_as_float(ac[x + 32]));
                        sc[x] = s2.x;
                        sc[x + 32] = s2.y;
                    }
                }
                const int jlim = p.M + i - t * BN;  // keys jj > jlim are masked
                if (jlim < BN - 1) {
#pragma unroll
                    for (int x = 0; x < 64; ++x)
                        if (x > jlim) sc[x] = -INFINITY;
                }
#pragma unroll
                for (int x = 0; x < 64; ++x) sc[x] = ex2(sc[x] - lse);  // P
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->dp_full, gt & 1, kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
                tc_fence_after();
                uint32_t w[32];
                {
                    uint32_t dp[64];
                    tmem_ld32(tmem + lane_off + QA_COL_DP, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
                    tmem_ld32(tmem + lane_off + QA_COL_DP + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    warp_arrive(&sh->dp_free);
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        w[x] = pack_bf16x2(sc[2 * x] * (__uint_as_float(dp[2 * x]) - Dv),
                                           sc[2 * x + 1] * (__uint_as_float(dp[2 * x + 1]) - Dv));
                }
                __syncwarp();  // every lane's scratch reads precede the dS rows
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t a = ds_tile + db * SZ_Q + ii * 128 + ((c8 ^ (ii & 7)) << 4);
                    if (QA_SMEM_IN(a, 16, 702))
                        st_shared_v4(a, w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
                }
                fence_proxy_async_smem();
                warp_arrive(&sh->ds_full[db]);
            }
            gring += it.nt + 2;
        }
        tc_fence_before();
    } else if (warp == 4) {
        // ------------------------------------------ score issuer: AC, band, dP
        const uint32_t leader = elect_one();
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kDevTimeoutMma, abort, p.status));
            return ok;
        };
        const uint64_t dQu = smem_desc_sw128(s_base + QA_OFF_QU, 16, 1024);
        const uint64_t dQv = smem_desc_sw128(s_base + QA_OFF_QV, 16, 1024);
        const uint64_t dDO = smem_desc_sw128(s_base + QA_OFF_DO, 16, 1024);
        const uint64_t dKV = smem_desc_sw128(s_base + QA_OFF_KV, 16, 1024);
        const uint64_t dR = smem_desc_sw128(s_base + QA_OFF_R, 16, 1024);
        constexpr uint32_t U_T = SZ_T >> 4, U_Q = SZ_Q >> 4;
        int gt = 0, rbox = 0, gring = 0;
        QaItem it;
        for (int k = 0; ok && qa_item(p, k, it); ++k) {
            wait(&sh->qa_full, k & 1);
            wait(&sh->qv_full, k & 1);
            const uint64_t aQv = dQv;
            for (int t = 0; ok && t < it.nt; ++t) {
                const int gt_t = gt + t;
                const int st = gt_t % QA_KV;
                const bool last = t == it.nt - 1;
                // AC(t) and the band slots tile t is the first to read: S and
                // the ring position of slot t+2 (slot t-1's) are free once
                // the softmax has read tile t-1
                if (gt_t > 0) wait(&sh->s_free, (gt_t - 1) & 1);
                wait(&sh->kv_full[st], (gt_t / QA_KV) & 1);
                for (int s = (t == 0 ? 0 : t + 2); ok && s <= t + 2; ++s) {
                    const int rb = rbox + (s >> 1);
                    if ((s & 1) == 0 || s == 1) wait(&sh->r_full[rb % QA_RB], (rb / QA_RB) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + QA_COL_RING + 64 * ((gring + s) % QA_RING);
                    const uint64_t bR = dR + (rb % QA_RB) * U_Q + (s & 1) * U_T;
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        mma_ss_elect(d, aQv + 2 * kk, bR + 2 * kk, IDESC_N64, kk > 0, leader);
                    // the box's last position slot (or the item's)
                    if (leader && ((s & 1) || s == it.nt + 1)) mma_commit(&sh->r_empty[rb % QA_RB]);
                }
                if (!ok) break;
                tc_fence_after();
                const uint64_t bK = dKV + st * 2 * U_T;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk)
                    mma_ss_elect(tmem + QA_COL_S, dQu + 2 * kk, bK + 2 * kk, IDESC_N64, kk > 0, leader);
                if (leader) {
                    mma_commit(&sh->s_full);
                    if (last) mma_commit(&sh->qv_empty);
                }
                // dP(t) once the softmax has read dP(t-1)
                if (gt_t > 0) wait(&sh->dp_free, (gt_t - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t bV = bK + U_T;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk)
                    mma_ss_elect(tmem + QA_COL_DP, dDO + 2 * kk, bV + 2 * kk, IDESC_N64, kk > 0, leader);
                if (leader) {
                    mma_commit(&sh->dp_full);
                    mma_commit(&sh->kv_empty[st]);
                    if (last) mma_commit(&sh->qa_empty);
                }
            }
            gt += it.nt;
            rbox += (it.nt + 3) >> 1;
            gring += it.nt + 2;
        }
        if (leader) mma_commit(&sh->drain[0]);
        drain_wait(&sh->drain[0], 0, p.status);
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            int kvc = 0;
            QaItem it;
            for (int k = 0; ok && qa_item(p, k, it); ++k) {
                if (k > 0 && !mbar_wait(&sh->qa_empty, (k - 1) & 1, kDevTimeoutProducer, abort, p.status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&sh->qa_full, 2 * SZ_Q);
                tma_load_3d(smem + QA_OFF_QU, &tmQu, &sh->qa_full, 0, it.i0, it.bh);
                tma_load_3d(smem + QA_OFF_DO, &tmDO, &sh->qa_full, 0, it.i0, it.bh);
                if (k > 0 && !mbar_wait(&sh->qv_empty, (k - 1) & 1, kDevTimeoutProducer, abort, p.status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&sh->qv_full, SZ_Q);
                tma_load_3d(smem + QA_OFF_QV, &tmQv, &sh->qv_full, 0, it.i0, it.bh);
                for (int t = 0; t < it.nt; ++t, ++kvc) {
                    const int s = kvc % QA_KV;
                    if (kvc >= QA_KV && !mbar_wait(&sh->kv_empty[s], ((kvc / QA_KV) & 1) ^ 1,
                                                   kDevTimeoutProducer, abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&sh->kv_full[s], 2 * SZ_T);
                    uint8_t* dst = smem + QA_OFF_KV + s * 2 * SZ_T;
                    tma_load_3d(dst, &tmK, &sh->kv_full[s], 0, t * BN, it.bh);
                    tma_load_3d(dst + SZ_T, &tmV, &sh->kv_full[s], 0, t * BN, it.bh);
                }
            }
            for (int c = kvc - QA_KV; c < kvc; ++c)
                if (c >= 0) drain_wait(&sh->kv_full[c % QA_KV], (c / QA_KV) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == 11) {
        // -------------------------------------------- TMA producer: R boxes
        if (lane == 0) {
            bool ok = true;
            int rc = 0;
            QaItem it;
            for (int k = 0; ok && qa_item(p, k, it); ++k) {
                const int nb = (it.nt + 3) >> 1;
                for (int b = 0; b < nb; ++b, ++rc) {
                    const int s = rc % QA_RB;
                    if (rc >= QA_RB && !mbar_wait(&sh->r_empty[s], ((rc / QA_RB) & 1) ^ 1, kDevTimeoutProducer,
                                                  abort, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&sh->r_full[s], SZ_Q);
                    tma_load_2d(smem + QA_OFF_R + s * SZ_Q, &tmR, &sh->r_full[s], it.h * DH, it.rbase + 128 * b);
                }
            }
            for (int c = rc - QA_RB; c < rc; ++c)
                if (c >= 0) drain_wait(&sh->r_full[c % QA_RB], (c / QA_RB) & 1, p.status);
        }
        __syncwarp();
    } else if (warp < 10) {
        // --------------------------------------------- band scatter, dR, dq
        // warp w serves TMEM lane quarter w % 4: query row ii = 32 (w%4) +
        // lane of the scatter and of dq, band row ii of each dR pair
        const int wq = warp & 3;
        const int ii = 32 * wq + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t g_base = s_base + QA_OFF_G;
        const int o = 127 - ii;      // band column of key 0 of tile 0
        const int e = o & 7;         // columns of the first chunk before it
        const int a0 = o >> 3;       // chunk of the row's first value in tile 0
        bool ok = true;
        int gt = 0, ndr = 0, gslot = 0;
        QaItem it;
        for (int k = 0; ok && qa_item(p, k, it); ++k) {
            const int nb = (it.nt + 3) >> 1;
            uint32_t cw[4] = {0u, 0u, 0u, 0u};  // previous tile's last 8 dS values of the row
            int next_dr = 0;
            for (int t = 0; t < it.nt; ++t, ++gt) {
                const bool last = t == it.nt - 1;
                // one barrier per dS buffer: the softmax can finish tile gt+1
                // before this warp has seen tile gt, never tile gt+2
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->ds_full[gt & 1], (gt >> 1) & 1, kDevTimeoutSoftmax,
                                                       abort, p.status));
                if (!ok) break;
                uint32_t w[32];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t a = ds_tile + (gt & 1) * SZ_Q + ii * 128 + ((c8 ^ (ii & 7)) << 4);
                    if (QA_SMEM_IN(a, 16, 708)) ld_shared_v4u(a, w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
                }
                warp_arrive(&sh->ds_read[gt & 1]);
                // the G positions of slots t .. t+2 are free once the MMAs
                // after the previous tile's scatter completed
                if (gt > 0)
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&sh->post, (gt - 1) & 1, kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
                // leading zero chunks before tile 0's first chunk, the tile's
                // 8 chunks, and after the last tile its remaining values and
                // the trailing zero chunks up to the end of slot nt+1
                if (t == 0) {
                    for (int ch = 0; ch < a0; ++ch) {
                        const uint32_t a = g_chunk_addr(g_base, gslot, ch, ii);
                        if (QA_SMEM_IN(a, 16, 703)) st_shared_v4(a, 0u, 0u, 0u, 0u);
                    }
                }
                {
                    uint32_t ow[32];
                    g_align(cw, w, e, ow);
#pragma unroll
                    for (int kc = 0; kc < 8; ++kc) {
                        const uint32_t a = g_chunk_addr(g_base, gslot, 8 * t + a0 + kc, ii);
                        if (QA_SMEM_IN(a, 16, 704))
                            st_shared_v4(a, ow[4 * kc], ow[4 * kc + 1], ow[4 * kc + 2], ow[4 * kc + 3]);
                    }
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) cw[x] = w[28 + x];
                if (last) {
                    // chunk 8 of the last tile: its last e values, then zeros
                    uint32_t ow[32];
                    const uint32_t zw[32] = {};
                    g_align(cw, zw, e, ow);
                    const int ch0 = 8 * (t + 1) + a0;
                    const int ch_end = 8 * (it.nt + 2);
                    for (int ch = ch0; ch < ch_end; ++ch) {
                        const uint32_t a = g_chunk_addr(g_base, gslot, ch, ii);
                        const bool first = ch == ch0;
                        if (QA_SMEM_IN(a, 16, 705))
                            st_shared_v4(a, first ? ow[0] : 0u, first ? ow[1] : 0u, first ? ow[2] : 0u,
                                         first ? ow[3] : 0u);
                    }
                }
                fence_proxy_async_smem();
                warp_arrive(&sh->g_full);
                // the dR pairs this tile completes
                const int dr_end = last ? nb : (t + 1) >> 1;
                for (; next_dr < dr_end; ++next_dr, ++ndr) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&sh->dr_full, ndr & 1, kDevTimeoutSoftmax, abort, p.status));
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem + lane_off + QA_COL_DR, r0);
                    tmem_ld32(tmem + lane_off + QA_COL_DR + 32, r1);
                    tmem_wait_ld();
                    tc_fence_before();
                    warp_arrive(&sh->dr_free);
                    const int slot = 2 * next_dr + (ii >> 6);
                    const int row = it.rbase + 128 * next_dr + ii;
                    if (slot <= it.nt + 1 && row >= 0 && row < p.K &&
                        TXL_BOUNDS((size_t)row * p.H + it.h < (size_t)p.K * p.H, 707, row)) {
                        float* dst = p.dr + ((size_t)row * p.H + it.h) * DH;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            red_add_v4(dst + 4 * c, kLn2 * __uint_as_float(r0[4 * c]),
                                       kLn2 * __uint_as_float(r0[4 * c + 1]), kLn2 * __uint_as_float(r0[4 * c + 2]),
                                       kLn2 * __uint_as_float(r0[4 * c + 3]));
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            red_add_v4(dst + 32 + 4 * c, kLn2 * __uint_as_float(r1[4 * c]),
                                       kLn2 * __uint_as_float(r1[4 * c + 1]), kLn2 * __uint_as_float(r1[4 * c + 2]),
                                       kLn2 * __uint_as_float(r1[4 * c + 3]));
                    }
                }
                if (!ok) break;
            }
            if (!ok) break;
            // ------------------------------------------ dq, du, dv_bias
            ok = __all_sync(0xffffffffu, mbar_wait(&sh->dq_done, k & 1, kDevTimeoutSoftmax, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            // two halves of 32 columns: dq = scale (dq_c + dq_p) per row, and
            // the warp's column sums of scale dq_c, scale dq_p into du, dv_bias
            // (rows past L hold dS = 0: their dq_c, dq_p are zero)
            const int i = it.i0 + ii;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t rc[32], rp[32];
                tmem_ld32(tmem + lane_off + QA_COL_DQC + 32 * c, rc);
                tmem_ld32(tmem + lane_off + QA_COL_DQP + 32 * c, rp);
                tmem_wait_ld();
                if (c == 1) {
                    tc_fence_before();
                    warp_arrive(&sh->dq_free);
                }
                float vc[32], vp[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    vc[x] = p.scale * __uint_as_float(rc[x]);
                    vp[x] = p.scale * __uint_as_float(rp[x]);
                }
                if (i < p.L && TXL_BOUNDS(it.bh < p.B * p.H, 706, it.bh)) {
                    float4* dst = reinterpret_cast<float4*>(p.dq + ((size_t)it.bh * p.L + i) * DH + 32 * c);
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        dst[x] = make_float4(vc[4 * x] + vp[4 * x], vc[4 * x + 1] + vp[4 * x + 1],
                                             vc[4 * x + 2] + vp[4 * x + 2], vc[4 * x + 3] + vp[4 * x + 3]);
                }
                atomicAdd(p.du + it.h * DH + 32 * c + lane, warp_sum32(vc));
                atomicAdd(p.dvb + it.h * DH + 32 * c + lane, warp_sum32(vp));
            }
            gslot += qa_slots(it.nt);
        }
        tc_fence_before();
    } else if (warp == 10) {
        // --------------------------------------- gradient issuer: dq_c, dq_p, dR
        const uint32_t leader = elect_one();
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kDevTimeoutMma, abort, p.status));
            return ok;
        };
        // MN-major views (d_h contiguous): K and R as the B of dq; G read
        // transposed and (q+v)c as the A and B of dR
        const uint64_t dKmn = smem_desc_sw128(s_base + QA_OFF_KV, 8192, 1024);
        const uint64_t dRmn = smem_desc_sw128(s_base + QA_OFF_R, 8192, 1024);
        const uint64_t dDS = smem_desc_sw128(s_base + QA_OFF_DS, 16, 1024);
        const uint64_t dG = smem_desc_sw128(s_base + QA_OFF_G, 16, 1024);
        const uint64_t dGmn = smem_desc_sw128(s_base + QA_OFF_G, SZ_Q, 1024);
        const uint64_t dQvmn = smem_desc_sw128(s_base + QA_OFF_QV, 8192, 1024);
        constexpr uint32_t U_T = SZ_T >> 4, U_Q = SZ_Q >> 4;
        int gt = 0, rbox = 0, gslot = 0, ndr = 0;
        QaItem it;
        for (int k = 0; ok && qa_item(p, k, it); ++k) {
            const int nb = (it.nt + 3) >> 1;
            const uint64_t bQv = dQvmn;
            int next_dr = 0;
            for (int t = 0; ok && t < it.nt; ++t) {
                const int gt_t = gt + t;
                const int st = gt_t % QA_KV;
                const bool last = t == it.nt - 1;
                // dq_c(t) once the dS tile is in shared memory (the item's
                // first one overwrites dq_c: the flush warps have read the
                // previous item's)
                wait(&sh->ds_full[gt_t & 1], (gt_t >> 1) & 1);
                if (t == 0 && k > 0) wait(&sh->dq_free, (k - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t bKmn = dKmn + st * 2 * U_T;
                const uint64_t aDS = dDS + (gt_t & 1) * U_Q;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ss_elect(tmem + QA_COL_DQC, aDS + 2 * kk, bKmn + kk * 128, IDESC_N64_BMN,
                                 (kk > 0 || t > 0) ? 1u : 0u, leader);
                if (leader) {
                    mma_commit(&sh->dqc_done[gt_t & 1]);
                    mma_commit(&sh->kv_empty[st]);
                }
                // dq_p of the band slots complete after tile t and dR of the
                // complete slot pairs, once the tile's scatter is in G
                wait(&sh->g_full, gt_t & 1);
                if (!ok) break;
                tc_fence_after();
                const int s_hi = last ? it.nt + 1 : t;
                for (int s = t; s <= s_hi; ++s) {
                    const int rb = rbox + (s >> 1);
                    const uint64_t aG = dG + ((gslot + s) & (QA_G - 1)) * U_Q;
                    const uint64_t bR = dRmn + (rb % QA_RB) * U_Q + (s & 1) * U_T;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ss_elect(tmem + QA_COL_DQP, aG + 2 * kk, bR + kk * 128, IDESC_N64_BMN,
                                     (kk > 0 || s > 0) ? 1u : 0u, leader);
                    // the box's last slot (or the item's)
                    if (leader && ((s & 1) || s == it.nt + 1)) mma_commit(&sh->r_empty[rb % QA_RB]);
                }
                const int dr_end = last ? nb : (t + 1) >> 1;
                for (; ok && next_dr < dr_end; ++next_dr) {
                    // G slots 2b, 2b+1 (adjacent ring positions) read
                    // transposed: M = 128 band rows, K = 128 query rows
                    if (ndr > 0) wait(&sh->dr_free, (ndr - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t aG = dGmn + ((gslot + 2 * next_dr) & (QA_G - 1)) * U_Q;
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ss_elect(tmem + QA_COL_DR, aG + kk * 128, bQv + kk * 128, IDESC_N64_ABMN, kk > 0,
                                     leader);
                    if (leader) mma_commit(&sh->dr_full);
                    ++ndr;
                }
                if (!ok) break;
                if (leader) {
                    mma_commit(&sh->post);
                    if (last) {
                        mma_commit(&sh->qv_empty);
                        mma_commit(&sh->dq_done);
                    }
                }
            }
            gt += it.nt;
            rbox += nb;
            gslot += qa_slots(it.nt);
        }
        if (leader) mma_commit(&sh->drain[1]);
        drain_wait(&sh->drain[1], 0, p.status);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// --------------------------------------------------------------------------
// attn_bwd_kv_kernel: dK, dV.
//
// Per step (query tile of the item; global step counter gs across items):
//   issuer:  [scores] AC = (q+u)c K^T (N = 128) -> S; band = (q+v)c Rb^T with
//                     the 256 R rows rb0 .. rb0+255 (rb0 = j0 + L - i0 - 128;
//                     pair (ii, jj) reads band column 127 - ii + jj) -> BAND
//            [dP]     dP = dout V^T (N = 128) -> S, once S has been read
//            [dV]     dV += P^T dout, once P is in shared memory
//            [dK]     dK += dS^T (q+u)c, once dS is in shared memory
//   softmax: thread (row ii, key half hh) reads AC columns 64 hh .. and band
//            columns 96 - 32 wq + 64 hh .. (96 of them), shifts the band,
//            P = 2^(s - lse) into the P buffer (row ii of half hh: the
//            transposed A of dV), then dP, dS = P (dP - D) into the same
//            place once the dV MMA has read P.
// Issue order: [scores](first), then per step [dP], [dV], [scores](next step,
// possibly of the next item), [dK].
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(bw::KB_THREADS, 1)
attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQu, const __grid_constant__ CUtensorMap tmQv,
                   const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmR,
                   const BwdParams p) {
    using namespace bw;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    KbShared* sh = reinterpret_cast<KbShared*>(smem + KB_OFF_BAR);
    const uint32_t s_base = smem_u32(smem);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (warp == 8) {
        tmem_alloc(&sh->tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 9 && lane == 0) {
        tma_prefetch_desc(&tmQu);
        tma_prefetch_desc(&tmQv);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmR);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh->kv_full[s], 1);
            mbar_init(&sh->kv_empty[s], 1);
            mbar_init(&sh->q_full[s], 1);
            mbar_init(&sh->q_empty[s], 1);
        }
        mbar_init(&sh->qv_full, 1);
        mbar_init(&sh->qv_empty, 1);
        mbar_init(&sh->r_full, 1);
        mbar_init(&sh->r_empty, 1);
        mbar_init(&sh->s_full, 1);
        mbar_init(&sh->s_free, 8);
        mbar_init(&sh->dp_full, 1);
        mbar_init(&sh->dp_free, 8);
        mbar_init(&sh->pt_full, 8);
        mbar_init(&sh->pv_done, 1);
        mbar_init(&sh->ds_full, 8);
        mbar_init(&sh->post, 1);
        mbar_init(&sh->dkv_done, 1);
        mbar_init(&sh->drain, 1);
        sh->abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;

    if (warp < 8) {
        // ---------------------------------------------------------- softmax
        const int wq = warp & 3;
        const int hh = warp >> 2;                // key half of the block
        const int ii = 32 * wq + lane;           // query row within the step
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t p_half = s_base + KB_OFF_P + hh * SZ_Q;
        const uint32_t t_ld = p_half + wq * 4096 + 4 * lane;
        const uint32_t t_st = t_ld - 128u * (uint32_t)(31 - lane);
        const int c0 = 96 - 32 * wq + 64 * hh;  // first band column the warp reads
        bool ok = true;
        int gs = 0;
        KbItem it;
        for (int k = 0; ok && kb_item(p, k, it); ++k) {
            for (int q = 0; q < it.nsteps; ++q, ++gs) {
                const int i0 = (it.qlo + q) * BM;
                const int i = i0 + ii;
                float lse = INFINITY, Dv = 0.f;
                if (i < p.L) {
                    const float2 st = p.stats[(size_t)it.bh * p.L + i];
                    lse = st.x;
                    Dv = st.y;
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->s_full, gs & 1, kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
                tc_fence_after();
                float sc[64];
                {
                    // the band first (packed and stored to the shift scratch),
                    // then AC: the two are never held in registers together
                    uint32_t hp[64];
                    {
                        uint32_t bwv[96];
#pragma unroll
                        for (int kc = 0; kc < 3; ++kc)
                            tmem_ld32(tmem + lane_off + KB_COL_BAND + c0 + 32 * kc,
                                      *reinterpret_cast<uint32_t(*)[32]>(&bwv[32 * kc]));
                        tmem_wait_ld();
#pragma unroll
                        for (int K = 0; K < 64; ++K)
                            hp[K] = pack_f16x2_sat(__uint_as_float(bwv[K]), __uint_as_float(bwv[K + 32]));
                    }
                    // the P / dS buffer is free once the previous dK MMA completed
                    if (gs > 0)
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait(&sh->post, (gs - 1) & 1, kDevTimeoutSoftmax, abort, p.status));
                    if (!ok) break;
                    __syncwarp();
                    if (!KB_SMEM_IN(t_ld, 128 * 31 + 4, 711)) break;
                    st_shift_all<0>(31 - lane, t_st, *reinterpret_cast<uint32_t(*)[32]>(&hp[0]),
                                    *reinterpret_cast<uint32_t(*)[32]>(&hp[32]));
                    uint32_t ac[64];
                    tmem_ld32(tmem + lane_off + KB_COL_S + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&ac[0]));
                    tmem_ld32(tmem + lane_off + KB_COL_S + 64 * hh + 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&ac[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    warp_arrive(&sh->s_free);
                    float win[32];
                    ld_shift_all<0>(t_ld, win);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const float2 s2 = add_h2_f32(__float_as_uint(win[x]), __uint_as_float(ac[x]),
                                                     __uint_as_float(ac[x + 32]));
                        sc[x] = s2.x;
                        sc[x + 32] = s2.y;
                    }
                }
                const int jlim = p.M + i - it.j0 - 64 * hh;  // keys x > jlim of the half are masked
                if (jlim < 63) {
#pragma unroll
                    for (int x = 0; x < 64; ++x)
                        if (x > jlim) sc[x] = -INFINITY;
                }
#pragma unroll
                for (int x = 0; x < 64; ++x) sc[x] = ex2(sc[x] - lse);  // P
                __syncwarp();  // every lane's scratch reads precede the P rows
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t a = p_half + ii * 128 + ((c8 ^ (ii & 7)) << 4);
                    if (KB_SMEM_IN(a, 16, 712))
                        st_shared_v4(a, pack_bf16x2(sc[8 * c8], sc[8 * c8 + 1]),
                                     pack_bf16x2(sc[8 * c8 + 2], sc[8 * c8 + 3]),
                                     pack_bf16x2(sc[8 * c8 + 4], sc[8 * c8 + 5]),
                                     pack_bf16x2(sc[8 * c8 + 6], sc[8 * c8 + 7]));
                }
                fence_proxy_async_smem();
                warp_arrive(&sh->pt_full);
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->dp_full, gs & 1, kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
                tc_fence_after();
                uint32_t w[32];
                {
                    uint32_t dp[64];
                    tmem_ld32(tmem + lane_off + KB_COL_S + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
                    tmem_ld32(tmem + lane_off + KB_COL_S + 64 * hh + 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    warp_arrive(&sh->dp_free);
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        w[x] = pack_bf16x2(sc[2 * x] * (__uint_as_float(dp[2 * x]) - Dv),
                                           sc[2 * x + 1] * (__uint_as_float(dp[2 * x + 1]) - Dv));
                }
                // dS overwrites P once the dV MMA has read it
                ok = __all_sync(0xffffffffu, mbar_wait(&sh->pv_done, gs & 1, kDevTimeoutSoftmax, abort, p.status));
                if (!ok) break;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t a = p_half + ii * 128 + ((c8 ^ (ii & 7)) << 4);
                    if (KB_SMEM_IN(a, 16, 713)) st_shared_v4(a, w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
                }
                fence_proxy_async_smem();
                warp_arrive(&sh->ds_full);
            }
            if (!ok) break;
            // ------------------------------------------------ dK or dV rows
            ok = __all_sync(0xffffffffu, mbar_wait(&sh->dkv_done, k & 1, kDevTimeoutSoftmax, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            const int j = it.j0 + ii;  // key row = TMEM lane
            float* dst = (hh == 0 ? p.dk : p.dv) + ((size_t)it.bh * p.K + j) * DH;
            const float f = hh == 0 ? kLn2 : 1.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + (hh == 0 ? KB_COL_DK : KB_COL_DV) + 32 * c, r);
                tmem_wait_ld();
                if (j < p.K && TXL_BOUNDS(it.bh < p.B * p.H, 714, it.bh)) {
                    float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        d4[x] = make_float4(f * __uint_as_float(r[4 * x]), f * __uint_as_float(r[4 * x + 1]),
                                            f * __uint_as_float(r[4 * x + 2]), f * __uint_as_float(r[4 * x + 3]));
                }
            }
            tc_fence_before();
        }
        tc_fence_before();
    } else if (warp == 8) {
        // ------------------------------------------------------- MMA issuer
        const uint32_t leader = elect_one();
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kDevTimeoutMma, abort, p.status));
            return ok;
        };
        constexpr uint32_t U_Q = SZ_Q >> 4;
        const uint64_t dKf = smem_desc_sw128(s_base + KB_OFF_KV, 16, 1024);      // + 2 U_Q * buffer
        const uint64_t dQu = smem_desc_sw128(s_base + KB_OFF_ST, 16, 1024);      // + 2 U_Q * stage
        const uint64_t dQumn = smem_desc_sw128(s_base + KB_OFF_ST, 8192, 1024);  // + 2 U_Q * stage
        const uint64_t dQv = smem_desc_sw128(s_base + KB_OFF_QV, 16, 1024);
        const uint64_t dRb = smem_desc_sw128(s_base + KB_OFF_R, 16, 1024);
        const uint64_t dPmn = smem_desc_sw128(s_base + KB_OFF_P, SZ_Q, 1024);
        // the position band of step gs_q: once the band of the step before
        // has been read (its (q+v)c and R loaded)
        auto band = [&](int gs_q) {
            wait(&sh->qv_full, gs_q & 1);
            wait(&sh->r_full, gs_q & 1);
            if (gs_q > 0) wait(&sh->s_free, (gs_q - 1) & 1);
            if (!ok) return;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk)
                mma_ss_elect(tmem + KB_COL_BAND, dQv + 2 * kk, dRb + 2 * kk, IDESC_N256, kk > 0, leader);
            if (leader) {
                mma_commit(&sh->qv_empty);
                mma_commit(&sh->r_empty);
            }
        };
        // AC of step gs_q into S once dP of the step before has been read;
        // the step's scores are then complete
        auto ac = [&](int kitem, int gs_q) {
            const int stg = gs_q & 1;
            wait(&sh->kv_full[kitem & 1], (kitem >> 1) & 1);
            wait(&sh->q_full[stg], (gs_q >> 1) & 1);
            if (gs_q > 0) wait(&sh->dp_free, (gs_q - 1) & 1);
            if (!ok) return;
            tc_fence_after();
            const uint64_t bK = dKf + (kitem & 1) * 2 * U_Q;
            const uint64_t aQ = dQu + stg * 2 * U_Q;
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk)
                mma_ss_elect(tmem + KB_COL_S, aQ + 2 * kk, bK + 2 * kk, IDESC_N128, kk > 0, leader);
            if (leader) mma_commit(&sh->s_full);
        };
        int gs = 0;
        KbItem it, nx;
        bool have = kb_item(p, 0, it);
        if (have) {
            band(0);
            ac(0, 0);
        }
        for (int k = 0; ok && have; ++k) {
            const bool have_next = kb_item(p, k + 1, nx);
            for (int q = 0; ok && q < it.nsteps; ++q) {
                const int gs_q = gs + q;
                const int stg = gs_q & 1;
                const bool more = q + 1 < it.nsteps || have_next;  // a next step exists
                // dP into S once the scores have been read
                wait(&sh->s_free, gs_q & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t aDO = dQu + stg * 2 * U_Q + U_Q;
                const uint64_t bV = dKf + (k & 1) * 2 * U_Q + U_Q;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk)
                    mma_ss_elect(tmem + KB_COL_S, aDO + 2 * kk, bV + 2 * kk, IDESC_N128, kk > 0, leader);
                if (leader) mma_commit(&sh->dp_full);
                // the next step's band as soon as this one's has been read
                if (more) band(gs_q + 1);
                // dV += P^T dout: A = P read transposed (M = 128 keys in two
                // 64-key halves 16 KB apart, K = 128 query rows)
                wait(&sh->pt_full, gs_q & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t bDOmn = dQumn + stg * 2 * U_Q + U_Q;
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk)
                    mma_ss_elect(tmem + KB_COL_DV, dPmn + kk * 128, bDOmn + kk * 128, IDESC_N64_ABMN,
                                 (q > 0 || kk > 0) ? 1u : 0u, leader);
                if (leader) mma_commit(&sh->pv_done);
                // the next step's AC (of the next item after this item's last step)
                if (q + 1 < it.nsteps)
                    ac(k, gs_q + 1);
                else if (have_next)
                    ac(k + 1, gs_q + 1);
                if (!ok) break;
                // dK += dS^T (q+u)c
                wait(&sh->ds_full, gs_q & 1);
                if (!ok) break;
                tc_fence_after();
                const uint64_t bQumn = dQumn + stg * 2 * U_Q;
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk)
                    mma_ss_elect(tmem + KB_COL_DK, dPmn + kk * 128, bQumn + kk * 128, IDESC_N64_ABMN,
                                 (q > 0 || kk > 0) ? 1u : 0u, leader);
                if (leader) {
                    mma_commit(&sh->post);
                    mma_commit(&sh->q_empty[stg]);
                    if (q == it.nsteps - 1) {
                        mma_commit(&sh->kv_empty[k & 1]);
                        mma_commit(&sh->dkv_done);
                    }
                }
            }
            gs += it.nsteps;
            it = nx;
            have = have_next;
        }
        if (leader) mma_commit(&sh->drain);
        drain_wait(&sh->drain, 0, p.status);
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // K/V per item (two buffers), (q+u)c and dout per step (two stages)
            bool ok = true;
            int gs = 0, nkv = 0;
            KbItem it;
            for (int k = 0; ok && kb_item(p, k, it); ++k) {
                const int b = k & 1;
                if (k >= 2 && !mbar_wait(&sh->kv_empty[b], ((k >> 1) & 1) ^ 1, kDevTimeoutProducer, abort, p.status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&sh->kv_full[b], 2 * SZ_Q);
                tma_load_3d(smem + KB_OFF_KV + b * 2 * SZ_Q, &tmK, &sh->kv_full[b], 0, it.j0, it.bh);
                tma_load_3d(smem + KB_OFF_KV + b * 2 * SZ_Q + SZ_Q, &tmV, &sh->kv_full[b], 0, it.j0, it.bh);
                ++nkv;
                for (int q = 0; q < it.nsteps; ++q, ++gs) {
                    const int s = gs & 1;
                    if (gs >= 2 && !mbar_wait(&sh->q_empty[s], ((gs >> 1) & 1) ^ 1, kDevTimeoutProducer, abort,
                                              p.status)) {
                        ok = false;
                        break;
                    }
                    const int i0 = (it.qlo + q) * BM;
                    mbar_expect_tx(&sh->q_full[s], 2 * SZ_Q);
                    tma_load_3d(smem + KB_OFF_ST + s * 2 * SZ_Q, &tmQu, &sh->q_full[s], 0, i0, it.bh);
                    tma_load_3d(smem + KB_OFF_ST + s * 2 * SZ_Q + SZ_Q, &tmDO, &sh->q_full[s], 0, i0, it.bh);
                }
            }
            for (int c = nkv - 2; c < nkv; ++c)
                if (c >= 0) drain_wait(&sh->kv_full[c & 1], (c >> 1) & 1, p.status);
            for (int c = gs - 2; c < gs; ++c)
                if (c >= 0) drain_wait(&sh->q_full[c & 1], (c >> 1) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------- TMA producer: (q+v)c and the R band per step
        if (lane == 0) {
            // (q+v)c and the 256-row R band per step (single buffers: the
            // band MMA is their only reader, early in the step)
            bool ok = true;
            int gs = 0;
            KbItem it;
            for (int k = 0; ok && kb_item(p, k, it); ++k) {
                for (int q = 0; q < it.nsteps; ++q, ++gs) {
                    if (gs >= 1 && (!mbar_wait(&sh->qv_empty, (gs - 1) & 1, kDevTimeoutProducer, abort, p.status) ||
                                    !mbar_wait(&sh->r_empty, (gs - 1) & 1, kDevTimeoutProducer, abort, p.status))) {
                        ok = false;
                        break;
                    }
                    const int i0 = (it.qlo + q) * BM;
                    const int rb0 = it.j0 + p.L - i0 - BM;
                    mbar_expect_tx(&sh->qv_full, SZ_Q);
                    tma_load_3d(smem + KB_OFF_QV, &tmQv, &sh->qv_full, 0, i0, it.bh);
                    mbar_expect_tx(&sh->r_full, 2 * SZ_Q);
                    tma_load_2d(smem + KB_OFF_R, &tmR, &sh->r_full, it.h * DH, rb0);
                    tma_load_2d(smem + KB_OFF_R + SZ_Q, &tmR, &sh->r_full, it.h * DH, rb0 + 128);
                }
            }
            if (gs >= 1) {
                drain_wait(&sh->qv_full, (gs - 1) & 1, p.status);
                drain_wait(&sh->r_full, (gs - 1) & 1, p.status);
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // Launched as a programmatic dependent of the query-major pass and
    // independent of it; this grid completes only after that pass completed,
    // so work after it in the stream sees every gradient.
    if (tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Per query row (8 threads, 8 columns each): the row's (lse, D = dout . out)
// from the forward's bf16 output and lse (log2 units), and the score operands
// (q+u)c, (q+v)c rounded to bf16 as the forward rounds them:
// (float(q) + float(bias)) * c.
__global__ void __launch_bounds__(256)
attn_bwd_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ ub,
                     const __nv_bfloat16* __restrict__ vb, const __nv_bfloat16* __restrict__ dout,
                     const __nv_bfloat16* __restrict__ out, const float* __restrict__ lse_in,
                     __nv_bfloat16* __restrict__ qu, __nv_bfloat16* __restrict__ qv, float2* __restrict__ stats,
                     int H, int L, float scale_log2, long long rows,
                     float4* __restrict__ dr, int n_dr4, float4* __restrict__ du, float4* __restrict__ dvb,
                     int n_b4) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long t = (long long)blockIdx.x * 256 + threadIdx.x;
    // dR, du and dv_bias are sums the query-major pass accumulates: zeroed here
    for (long long z = t; z < n_dr4; z += (long long)gridDim.x * 256) dr[z] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < n_b4) {
        du[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        dvb[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const long long row = t >> 3;
    const int c = (int)(t & 7);
    const bool live = row < rows;
    const long long rr = live ? row : 0;
    const int h = (int)(rr / L) % H;
    float d = 0.f;
    if (live) {
        float o[8];
        {
            const uint4 ov = *reinterpret_cast<const uint4*>(out + rr * bw::DH + 8 * c);
            const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(o2[e]);
                o[2 * e] = f.x;
                o[2 * e + 1] = f.y;
            }
        }
        const uint4 g = *reinterpret_cast<const uint4*>(dout + rr * bw::DH + 8 * c);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(g2[e]);
            d += f.x * o[2 * e] + f.y * o[2 * e + 1];
        }
    }
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 4);
    if (!live) return;
    const uint4 qq = *reinterpret_cast<const uint4*>(q + rr * bw::DH + 8 * c);
    const uint4 uu = *reinterpret_cast<const uint4*>(ub + (size_t)h * bw::DH + 8 * c);
    const uint4 vv = *reinterpret_cast<const uint4*>(vb + (size_t)h * bw::DH + 8 * c);
    const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qq);
    const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uu);
    const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vv);
    uint32_t ou[4], ov[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 qf = __bfloat1622float2(q2[e]), uf = __bfloat1622float2(u2[e]), vf = __bfloat1622float2(v2[e]);
        ou[e] = pack_bf16x2((qf.x + uf.x) * scale_log2, (qf.y + uf.y) * scale_log2);
        ov[e] = pack_bf16x2((qf.x + vf.x) * scale_log2, (qf.y + vf.y) * scale_log2);
    }
    *reinterpret_cast<uint4*>(qu + rr * bw::DH + 8 * c) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
    *reinterpret_cast<uint4*>(qv + rr * bw::DH + 8 * c) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
    if (c == 0) stats[rr] = make_float2(lse_in[rr], d);
}

// ---------------------------------------------------------------- host side
cudaError_t launch_attn_tc_bf16_lse(const void* q, const void* k, const void* v, const void* r, const void* ub,
                                    const void* vb, int B, int H, int L, int M, float scale, int lo_shift,
                                    void* out, float* lse, int* status, cudaStream_t stream);

namespace {
size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct BwdWs {
    __nv_bfloat16* out;  // the recomputed forward output (no saved state)
    float* lse;          // and its rows' log2-sum-exp
    __nv_bfloat16* qu;
    __nv_bfloat16* qv;
    float2* stats;
    size_t bytes;
};

BwdWs bwd_ws_layout(void* base, int B, int H, int L) {
    const size_t rows = (size_t)B * H * L;
    BwdWs w;
    char* c = static_cast<char*>(base);
    size_t off = 0;
    w.out = reinterpret_cast<__nv_bfloat16*>(c + off);
    off += up256(rows * bw::DH * 2);
    w.lse = reinterpret_cast<float*>(c + off);
    off += up256(rows * sizeof(float));
    w.qu = reinterpret_cast<__nv_bfloat16*>(c + off);
    off += up256(rows * bw::DH * 2);
    w.qv = reinterpret_cast<__nv_bfloat16*>(c + off);
    off += up256(rows * bw::DH * 2);
    w.stats = reinterpret_cast<float2*>(c + off);
    off += up256(rows * sizeof(float2));
    w.bytes = off;
    return w;
}

template <typename Kern>
cudaError_t launch_bwd_kernel(Kern kern, int grid, int threads, uint32_t smem, cudaStream_t stream, bool pdl,
                              const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const CUtensorMap& d,
                              const CUtensorMap& e, const CUtensorMap& f, const BwdParams& p) {
    // pdl: programmatic stream serialisation, the kernel may be scheduled
    // before the previous one in the stream completed (the kernel states
    // what it waits for)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a, b, c, d, e, f, p);
}
}  // namespace

size_t attn_bwd_tc_workspace_bytes(int B, int H, int L, int M) {
    (void)M;
    return bwd_ws_layout(nullptr, B, H, L).bytes;
}

// out / lse non-null: the forward's saved output and per-row log2-sum-exp
// (launch_attn_tc_bf16_lse); otherwise the forward is run first, writing
// both into the workspace.
cudaError_t launch_attn_bwd_tc(const void* q, const void* k, const void* v, const void* r, const void* ub,
                               const void* vb, const void* out, const float* lse, const void* dout, int B, int H,
                               int L, int M, float scale, float* dq, float* dk, float* dv, float* dr, float* du,
                               float* dvb, void* workspace, int* status, cudaStream_t stream) {
    using namespace bw;
    static PerDeviceOnce attrs;
    {
        const cudaError_t e = attrs.run([] {
            cudaError_t rr = cudaFuncSetAttribute(attn_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  QA_SMEM);
            if (rr == cudaSuccess)
                rr = cudaFuncSetAttribute(attn_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KB_SMEM);
            return rr;
        });
        if (e != cudaSuccess) return e;
    }
    const int K = M + L;
    const int n_bh = B * H;
    const int n_qtiles = (L + BM - 1) / BM;
    const BwdWs w = bwd_ws_layout(workspace, B, H, L);
    cudaError_t e = cudaSuccess;
    const bool saved = out && lse;
    if (!saved) {
        e = launch_attn_tc_bf16_lse(q, k, v, r, ub, vb, B, H, L, M, scale, 1 << 30, w.out, w.lse, status, stream);
        if (e != cudaSuccess) return e;
        out = w.out;
        lse = w.lse;
    }
    const long long rows = (long long)n_bh * L;
    const long long threads = rows * 8;
    const dim3 pgrid((unsigned)((threads + 255) / 256));
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* ubb = static_cast<const __nv_bfloat16*>(ub);
    const auto* vbb = static_cast<const __nv_bfloat16*>(vb);
    const auto* gb = static_cast<const __nv_bfloat16*>(dout);
    const auto* ob = static_cast<const __nv_bfloat16*>(out);
    const float sl = scale * 1.4426950408889634f;
    auto* dr4 = reinterpret_cast<float4*>(dr);
    auto* du4 = reinterpret_cast<float4*>(du);
    auto* dvb4 = reinterpret_cast<float4*>(dvb);
    const int n_dr4 = K * H * DH / 4, n_b4 = H * DH / 4;
    attn_bwd_prep_kernel<<<pgrid, 256, 0, stream>>>(qb, ubb, vbb, gb, ob, lse, w.qu, w.qv, w.stats, H, L, sl, rows,
                                                    dr4, n_dr4, du4, dvb4, n_b4);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap mQu, mQv, mDO, mKa, mVa, mKb, mVb, mR;
    {
        cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)L, (cuuint64_t)n_bh};
        cuuint64_t strides[2] = {(cuuint64_t)DH * 2, (cuuint64_t)L * DH * 2};
        cuuint32_t box[3] = {DH, BM, 1};
        if (!encode_bf16(&mQu, w.qu, 3, dims, strides, box) || !encode_bf16(&mQv, w.qv, 3, dims, strides, box) ||
            !encode_bf16(&mDO, dout, 3, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)DH, (cuuint64_t)K, (cuuint64_t)n_bh};
        cuuint64_t strides[2] = {(cuuint64_t)DH * 2, (cuuint64_t)K * DH * 2};
        cuuint32_t box_a[3] = {DH, BN, 1};
        cuuint32_t box_b[3] = {DH, 128, 1};
        if (!encode_bf16(&mKa, k, 3, dims, strides, box_a) || !encode_bf16(&mVa, v, 3, dims, strides, box_a) ||
            !encode_bf16(&mKb, k, 3, dims, strides, box_b) || !encode_bf16(&mVb, v, 3, dims, strides, box_b))
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)H * DH, (cuuint64_t)K};
        cuuint64_t strides[1] = {(cuuint64_t)H * DH * 2};
        cuuint32_t box[2] = {DH, 128};
        if (!encode_bf16(&mR, r, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    BwdParams p;
    p.B = B;
    p.H = H;
    p.L = L;
    p.M = M;
    p.K = K;
    p.n_qtiles = n_qtiles;
    p.n_ktiles = (K + 127) / 128;
    p.stats = w.stats;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dr = dr;
    p.du = du;
    p.dvb = dvb;
    p.scale = scale;
    p.status = status;
    const int sms = current_sm_count();
    p.n_items = n_bh * n_qtiles;
    // the query-major pass starts once the prep kernel completed (its
    // full-SM CTAs launched early would take the SMs the prep blocks still
    // need); the key-major pass may start on each SM it leaves
    e = launch_bwd_kernel(attn_bwd_q_kernel, p.n_items < sms ? p.n_items : sms, QA_THREADS, QA_SMEM, stream, false, mQu,
                          mQv, mDO, mKa, mVa, mR, p);
    if (e != cudaSuccess) return e;
    p.n_items = n_bh * p.n_ktiles;
    return launch_bwd_kernel(attn_bwd_kv_kernel, p.n_items < sms ? p.n_items : sms, KB_THREADS, KB_SMEM, stream, true, mQu,
                             mQv, mDO, mKb, mVb, mR, p);
}

TXL_BOUNDS_READER(bounds_word_attn_bwd_tc)

}  // namespace txl
