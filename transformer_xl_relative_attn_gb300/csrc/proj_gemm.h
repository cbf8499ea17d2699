// Internal interface of the projection GEMM (proj_gemm.cu) for the ABI layer.
#pragma once
#include <cuda_runtime.h>

namespace txl {

// Host description of one projection GEMM of a launch.  A row source is
// either row-major [B, T, K] (layout 0) or split into K / 64 heads,
// [B, K / 64, T, 64] (layout 1: an attention output feeding the next layer).
struct ProjGemm {
    const void* a_src;     // [B, Ta, K] (memory rows) or null when Ta = 0
    const void* b_src;     // [B, Tb, K]
    int Ta, Tb;
    int a_heads, b_heads;  // layouts of a_src and b_src
    const void* w;         // [N, K]
    int N;
    int T_out;             // rows per (batch row, head) of the outputs
    void* out[3];          // output column c -> out[c / d]
    int a_start;           // a_src is a ring of Ta rows starting at this row (a multiple of 128)
    int B = 0;             // batch rows of this problem (0: the launch's B)
    int plain = -1;        // -1: the launch's layout; 1: outputs row-major [rows, d]; 0: [B, H, T_out, dh]
};

// One launch of up to three projection GEMMs: out[c / d] <- rows of [a_src;
// b_src] (per batch row: Ta rows of a_src, then Tb rows of b_src) times w^T.
// plain = 1 writes row-major [rows, d] outputs, otherwise [B, H, T_out, dh]
// (a problem may override B and the layout).
// Requires Ta, Tb multiples of 128 (Ta may be 0), K a multiple of 64, N a
// multiple of 256, N / d <= 3.  cudaErrorInvalidValue: a tensor map could not
// be encoded.
cudaError_t launch_proj_gemm(const ProjGemm* gm, int n_gemm, int B, int K, int d, int H, int dh,
                             int plain, int* status, cudaStream_t stream);

// A plain Linear over rows of x (x_heads = 0: [B, T, K]; 1: [B, K / 64, T,
// 64]): out [B, T, N] = relu?(x W^T + bias) + resid (bias [N] and resid
// [B, T, N] may be null).  T a multiple of 128, K of 64, N of 256.
cudaError_t launch_linear(const void* x, int x_heads, int B, int T, int K, const void* w, int N,
                          const void* bias, const void* resid, int relu, void* out, int* status,
                          cudaStream_t stream);

}  // namespace txl
