// LayerNorm with a fused residual add, the normalisation of a decoder layer
// ("Transformer-XL模型 核心源码阅读笔记", RelPartialLearnableMultiHeadAttn.forward
// and PositionwiseFF: layer_norm(w + attn_out), layer_norm(inp + core_out);
// nn.LayerNorm: biased variance, eps inside the square root):
//
//   out[r] = (z - mean(z)) / sqrt(var(z) + eps) * gamma + beta,  z = x[r] (+ y[r])
//
// bf16 rows of d elements in and out, fp32 arithmetic.  One warp per row;
// each lane holds d / 32 elements as 16-byte vectors, so a row is read once
// and the mean and the variance (two passes over registers) need no second
// read.  out may be x or y itself (each warp reads its whole row first).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

template <int VPL>  // 16-byte vectors per lane: d = 256 * VPL
__global__ void __launch_bounds__(256) layer_norm_kernel(const __nv_bfloat16* x, const __nv_bfloat16* y,
                                                         const __nv_bfloat16* __restrict__ gamma,
                                                         const __nv_bfloat16* __restrict__ beta,
                                                         long long rows, float eps, __nv_bfloat16* out) {
    constexpr int d = 256 * VPL;
    // programmatic stream serialisation: let the next kernel launch, wait for
    // the previous one before touching global memory
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    float z[8 * VPL];
    const uint4* x4 = reinterpret_cast<const uint4*>(x + r * d);
    const uint4* y4 = y ? reinterpret_cast<const uint4*>(y + r * d) : nullptr;
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
        // vector index within the row: (c * 32 + lane) of d / 8
        const bool in_row = TXL_BOUNDS(c * 32 + lane < d / 8, 301, r * (d / 8) + c * 32 + lane);
        const uint4 a = in_row ? x4[c * 32 + lane] : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(a2[e]);
            z[8 * c + 2 * e] = f.x;
            z[8 * c + 2 * e + 1] = f.y;
        }
        if (y4 && in_row) {
            const uint4 b = y4[c * 32 + lane];
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(b2[e]);
                z[8 * c + 2 * e] += f.x;
                z[8 * c + 2 * e + 1] += f.y;
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8 * VPL; ++k) s += z[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s * (1.f / d);
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < 8 * VPL; ++k) {
        const float t = z[k] - mean;
        q = fmaf(t, t, q);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q * (1.f / d) + eps);
    const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
    const uint4* b4 = reinterpret_cast<const uint4*>(beta);
    uint4* o4 = reinterpret_cast<uint4*>(out + r * d);
#pragma unroll
    for (int c = 0; c < VPL; ++c) {
        if (!TXL_BOUNDS(c * 32 + lane < d / 8, 302, c * 32 + lane)) continue;
        const uint4 gv = __ldg(g4 + c * 32 + lane), bv = __ldg(b4 + c * 32 + lane);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
        const __nv_bfloat162* bb2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 gf = __bfloat1622float2(g2[e]), bf = __bfloat1622float2(bb2[e]);
            const __nv_bfloat162 o2 = __floats2bfloat162_rn(
                fmaf((z[8 * c + 2 * e] - mean) * rstd, gf.x, bf.x),
                fmaf((z[8 * c + 2 * e + 1] - mean) * rstd, gf.y, bf.y));
            w[e] = *reinterpret_cast<const uint32_t*>(&o2);
        }
        o4[c * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// d a multiple of 256 up to 2048 (else cudaErrorInvalidValue).
cudaError_t launch_layer_norm(const void* x, const void* y, const void* gamma, const void* beta,
                              long long rows, int d, float eps, void* out, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    const auto* xx = static_cast<const __nv_bfloat16*>(x);
    const auto* yy = static_cast<const __nv_bfloat16*>(y);
    const auto* gg = static_cast<const __nv_bfloat16*>(gamma);
    const auto* bb = static_cast<const __nv_bfloat16*>(beta);
    auto* oo = static_cast<__nv_bfloat16*>(out);
    const unsigned g = (unsigned)blocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (d) {
        case 256: return cudaLaunchKernelEx(&cfg, layer_norm_kernel<1>, xx, yy, gg, bb, rows, eps, oo);
        case 512: return cudaLaunchKernelEx(&cfg, layer_norm_kernel<2>, xx, yy, gg, bb, rows, eps, oo);
        case 768: return cudaLaunchKernelEx(&cfg, layer_norm_kernel<3>, xx, yy, gg, bb, rows, eps, oo);
        case 1024: return cudaLaunchKernelEx(&cfg, layer_norm_kernel<4>, xx, yy, gg, bb, rows, eps, oo);
        case 1536: return cudaLaunchKernelEx(&cfg, layer_norm_kernel<6>, xx, yy, gg, bb, rows, eps, oo);
        case 2048: return cudaLaunchKernelEx(&cfg, layer_norm_kernel<8>, xx, yy, gg, bb, rows, eps, oo);
        default: return cudaErrorInvalidValue;
    }
}

TXL_BOUNDS_READER(bounds_word_layer_norm)

}  // namespace txl
