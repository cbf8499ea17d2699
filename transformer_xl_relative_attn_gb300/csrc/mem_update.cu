// Tail_M memory roll, in place on the memory buffer.
//
// new[b, r] = [mem; h][b, r + L]  for r in [0, M)   ("Transformer-XL" notes,
// zty624, section "Segment-Level Recurrence": keep the newest M hidden states
// of [M_tau; H_tau]).  With L >= M every new row comes from h.  With L < M
// row r takes mem[r+L] while r+L < M, else h[r+L-M].
//
// In place without a workspace: rows r congruent to c modulo L form a chain
// c, c+L, c+2L, ...; row r reads row r+L, which belongs to the same chain, so
// chains are disjoint.  One thread walks one chain (for one 16-byte column of
// one batch row) in ascending order, loading a block of up to kChain sources
// into registers before it stores them, so every source is read before the
// store that overwrites it and the loads of a block are all in flight at once.
// Adjacent threads own adjacent 16-byte columns of the same row: every warp
// access is a contiguous 512-byte segment.
#include <cstdint>
#include <cuda_runtime.h>

namespace txl {

constexpr int kChain = 8;

template <typename V>
__global__ void __launch_bounds__(256) tail_m_kernel(V* __restrict__ mem, const V* __restrict__ hid,
                                                     int B, int L, int M, int rowv) {
    // rowv = row length in units of V; chains = min(L, M)
    const int chains = L < M ? L : M;
    const long long total = (long long)B * chains * rowv;
    long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total) return;
    const int col = (int)(t % rowv);
    const long long cb = t / rowv;
    const int c = (int)(cb % chains);
    const int b = (int)(cb / chains);
    V* mrow = mem + (size_t)b * M * rowv + col;
    const V* hrow = hid + (size_t)b * L * rowv + col;
    if (L >= M) {
        // one row per chain: new[c] = h[L - M + c]
        mrow[(size_t)c * rowv] = hrow[(size_t)(L - M + c) * rowv];
        return;
    }
    // chain rows r = c, c+L, ... < M
    for (int r0 = c; r0 < M; r0 += kChain * L) {
        V buf[kChain];
#pragma unroll
        for (int s = 0; s < kChain; ++s) {
            const int r = r0 + s * L;
            if (r < M) {
                const int src = r + L;
                buf[s] = src < M ? mrow[(size_t)src * rowv] : hrow[(size_t)(src - M) * rowv];
            }
        }
#pragma unroll
        for (int s = 0; s < kChain; ++s) {
            const int r = r0 + s * L;
            if (r < M) mrow[(size_t)r * rowv] = buf[s];
        }
    }
}

// Launches the roll with the widest unit the alignment allows.
cudaError_t launch_tail_m(void* mem, const void* hid, int B, int L, int M, size_t row_bytes,
                          cudaStream_t stream) {
    const int chains = L < M ? L : M;
    auto go = [&](auto tag) -> cudaError_t {
        using V = decltype(tag);
        const int rowv = (int)(row_bytes / sizeof(V));
        const long long total = (long long)B * chains * rowv;
        const int threads = 256;
        const long long blocks = (total + threads - 1) / threads;
        if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
        tail_m_kernel<V><<<(unsigned)blocks, threads, 0, stream>>>(
            static_cast<V*>(mem), static_cast<const V*>(hid), B, L, M, rowv);
        return cudaGetLastError();
    };
    const uintptr_t a = reinterpret_cast<uintptr_t>(mem) | reinterpret_cast<uintptr_t>(hid);
    if (row_bytes % 16 == 0 && a % 16 == 0) return go(uint4{});
    if (row_bytes % 8 == 0 && a % 8 == 0) return go(uint2{});
    if (row_bytes % 4 == 0 && a % 4 == 0) return go(uint32_t{});
    return go(uint16_t{});
}

}  // namespace txl
