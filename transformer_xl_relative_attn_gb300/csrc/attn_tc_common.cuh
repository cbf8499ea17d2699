// Helpers shared by the tensor-core attention kernels (forward and
// backward): bounded drains, warp arrivals, the exp2 and f16 packing
// primitives, the per-row band shift through shared memory, bulk stores and
// the tensor-map encoder.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

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

// One arrival per warp: every lane has issued its fences before the
// __syncwarp, which orders their writes before lane 0's release-arrive.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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

// Two f32 values rounded to f16 (finite: out-of-range values saturate to
// +-65504) in one 32-bit word, lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// (lo(h) + a, hi(h) + b): each f16 half of h added in f32 to an f32 value
__device__ __forceinline__ float2 add_h2_f32(uint32_t h, float a, float b) {
    float d, e;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
        : "=f"(d), "=f"(e)
        : "r"(h), "f"(a), "f"(b));
    return make_float2(d, e);
}

// TMA store of a shared-memory box to a 3-D tensor (out-of-range rows are
// clipped), committed as one bulk group of the issuing thread
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];\n\t"
        "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// the issuing thread's bulk stores have read their shared-memory source
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the issuing thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// one arrival on an mbarrier that counts as n
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n)
                 : "memory");
}

// (a.x + b.x, a.y + b.y) in one packed instruction
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}

// Per-row shift through shared memory.  A thread holds 64 consecutive band
// columns w0[0..31] | w1[0..31] of its row and needs window columns o .. o+31
// (o = 31 - lane).  It writes window column k to position k - o when k >= o
// and window column 32 + k to position k + 32 - o otherwise (for each k
// exactly one of the two lands in 0..31), then reads positions 0..31 back in
// order.  Position x of lane l is word 32 x + l of the warp's 4 KB scratch:
// each store and load of the warp touches 32 distinct banks, and a lane only
// ever touches its own words.  `base` is the lane's word of position 0 minus
// 128 o bytes.
template <int K>
__device__ __forceinline__ void st_shift_pair(int o, uint32_t base, uint32_t w0k, uint32_t w1k) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.le.s32 q, %0, %1;\n\t"
        "@q st.shared.b32 [%2+%3], %4;\n\t"
        "@!q st.shared.b32 [%2+%5], %6;\n\t}"
        ::"r"(o), "n"(K), "r"(base), "n"(128 * K), "r"(w0k), "n"(4096 + 128 * K), "r"(w1k)
        : "memory");
}
template <int K>
__device__ __forceinline__ float ld_shift(uint32_t base) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(base), "n"(128 * K) : "memory");
    return v;
}
template <int K>
__device__ __forceinline__ void st_shift_all(int o, uint32_t base, const uint32_t (&w0)[32],
                                             const uint32_t (&w1)[32]) {
    if constexpr (K < 32) {
        st_shift_pair<K>(o, base, w0[K], w1[K]);
        st_shift_all<K + 1>(o, base, w0, w1);
    }
}
template <int K>
__device__ __forceinline__ void ld_shift_all(uint32_t base, float (&win)[32]) {
    if constexpr (K < 32) {
        win[K] = ld_shift<K>(base);
        ld_shift_all<K + 1>(base, win);
    }
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, float (&v)[4]) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(addr)
                 : "memory");
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
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

inline bool encode_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                        const cuuint64_t* strides_bytes, const cuuint32_t* box,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                    strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


}  // namespace txl
