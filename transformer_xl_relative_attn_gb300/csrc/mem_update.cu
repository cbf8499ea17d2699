// Tail_M memory roll, in place on the memory buffer.
//
// new[b, r] = [mem; h][b, r + L]  for r in [0, M)   ("Transformer-XL" notes,
// zty624, section "Segment-Level Recurrence": keep the newest M hidden states
// of [M_tau; H_tau]).  With L >= M every new row comes from h.  With L < M
// row r takes mem[r+L] while r+L < M, else h[r+L-M].
//
// With ext_len > 0 the last ext_len rows of h are kept out of the memory
// ("Transformer-XL模型 核心源码阅读笔记", MemTransformerLM._update_mems: the
// cached span ends ext_len rows before the end of [mem; h]): the roll above
// with the first L - ext_len rows of h in place of h.
//
// In place without a workspace (details at each kernel).  Adjacent threads
// own adjacent vectors of a row, so every warp access is contiguous.
#include <cstdint>
#include <cuda_runtime.h>

#include "txl_device.cuh"

namespace txl {

constexpr int kChain = 16;  // sources of one chain in flight per thread
constexpr int kCopyUnroll = 4;  // vectors in flight per thread in the plain copy

// The roll kernels are launched with programmatic stream serialisation: each
// lets the next kernel of the stream launch at once and waits for the
// previous one to complete before its first global access, so back-to-back
// rolls do not pay a full launch gap each.
__device__ __forceinline__ void pdl_prologue() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, long long blocks, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// L >= M: every new row comes from h, and memory row r of batch b takes h row
// L-M+r, so the roll is one contiguous copy of M rows per batch row: element
// e of the flattened memory [B, M, row] is element (e / seg) * hstride + hoff
// + e % seg of h.  Each thread moves kCopyUnroll vectors spaced one block
// apart (coalesced per warp), all loads issued before the stores.
template <typename V, typename I>
__global__ void __launch_bounds__(256) tail_copy_kernel(V* __restrict__ mem, const V* __restrict__ hid,
                                                        I total, I seg, I hstride, I hoff) {
    pdl_prologue();
    const I base = (I)blockIdx.x * (256 * kCopyUnroll) + threadIdx.x;
    V buf[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const I e = base + (I)u * 256;
        if (e < total) {
            const I b = e / seg;
            const I hi = b * hstride + hoff + (e - b * seg);
            // hid holds total / seg batch rows of hstride vectors
            if (TXL_BOUNDS(hi >= 0 && hi < (total / seg) * hstride, 201, hi)) buf[u] = hid[hi];
        }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const I e = base + (I)u * 256;
        if (e < total && TXL_BOUNDS(e >= 0, 202, e)) mem[e] = buf[u];
    }
}

// L < M: rows r congruent to c modulo L form a chain c, c+L, c+2L, ...; row
// r reads row r+L of the same chain, so chains are disjoint and one thread
// walks one chain (for one vector column of one batch row) upwards, loading a
// block of kChain sources before storing them.
template <typename V, typename I>
__global__ void __launch_bounds__(256) tail_chain_kernel(V* __restrict__ mem, const V* __restrict__ hid,
                                                         int L, int M, I rowv, I total, I hstride) {
    pdl_prologue();
    const I t = (I)blockIdx.x * 256 + threadIdx.x;
    if (t >= total) return;
    const I col = t % rowv;
    const I cb = t / rowv;
    const int c = (int)(cb % (I)L);
    const I b = cb / (I)L;
    V* mrow = mem + b * (I)M * rowv + col;
    const V* hrow = hid + b * hstride + col;
    for (int r0 = c; r0 < M; r0 += kChain * L) {
        V buf[kChain];
#pragma unroll
        for (int s = 0; s < kChain; ++s) {
            const int r = r0 + s * L;
            if (r < M) {
                const int src = r + L;
                if (src < M) {
                    const I mi = (b * (I)M + src) * rowv + col;
                    if (TXL_BOUNDS(mi < (total / ((I)L * rowv)) * (I)M * rowv, 203, mi)) buf[s] = mrow[(I)src * rowv];
                } else {
                    const I hi = b * hstride + (I)(src - M) * rowv + col;
                    if (TXL_BOUNDS(hi < (total / ((I)L * rowv)) * hstride, 204, hi)) buf[s] = hrow[(I)(src - M) * rowv];
                }
            }
        }
#pragma unroll
        for (int s = 0; s < kChain; ++s) {
            const int r = r0 + s * L;
            if (r < M && TXL_BOUNDS((b * (I)M + r) * rowv + col < (total / ((I)L * rowv)) * (I)M * rowv, 205,
                                    (b * (I)M + r) * rowv + col))
                mrow[(I)r * rowv] = buf[s];
        }
    }
}

// Zeroes the memory rows of every batch row b with flags[b] != 0 (a batch
// row whose stream starts a new document; "Transformer-XL" notes, section
// "Batched Streams": the reset is per row).  mem is [B, rows, row]; one
// thread per vector.
template <typename V, typename I>
__global__ void __launch_bounds__(256) mem_reset_kernel(V* __restrict__ mem, const unsigned char* __restrict__ flags,
                                                        I per_b, I total) {
    const I e = (I)blockIdx.x * 256 + threadIdx.x;
    if (e >= total) return;
    if (TXL_BOUNDS(e / per_b < total / per_b, 206, e) && flags[e / per_b]) mem[e] = V{};
}

// Launches the roll with the widest vector the alignment allows and 32-bit
// index arithmetic whenever the element counts fit.  L rows of each batch
// row of hid take part; consecutive batch rows of hid are L_stride rows
// apart (L < L_stride when trailing rows are held back).
cudaError_t launch_tail_m(void* mem, const void* hid, int B, int L, int L_stride, int M,
                          size_t row_bytes, cudaStream_t stream) {
    if (L <= 0 || M <= 0) return cudaSuccess;  // nothing new enters, or no memory
    auto go = [&](auto tag) -> cudaError_t {
        using V = decltype(tag);
        const long long rowv = (long long)(row_bytes / sizeof(V));
        if (L >= M) {
            const long long seg = (long long)M * rowv, total = (long long)B * seg;
            const long long hsz = (long long)B * L_stride * rowv;
            const long long blocks = (total + 256 * kCopyUnroll - 1) / (256 * kCopyUnroll);
            if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
            if (hsz < 0x7FFFFFFFll - 256 * kCopyUnroll)
                return launch_pdl(tail_copy_kernel<V, int>, blocks, stream, static_cast<V*>(mem),
                                  static_cast<const V*>(hid), (int)total, (int)seg, (int)(L_stride * rowv),
                                  (int)((L - M) * rowv));
            return launch_pdl(tail_copy_kernel<V, long long>, blocks, stream, static_cast<V*>(mem),
                              static_cast<const V*>(hid), total, seg, L_stride * rowv, (L - M) * rowv);
        } else {
            const long long total = (long long)B * L * rowv;
            const long long msz = (long long)B * (M > L_stride ? M : L_stride) * rowv;
            const long long blocks = (total + 255) / 256;
            if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
            if (msz < 0x7FFFFFFFll - 256)
                return launch_pdl(tail_chain_kernel<V, int>, blocks, stream, static_cast<V*>(mem),
                                  static_cast<const V*>(hid), L, M, (int)rowv, (int)total, (int)(L_stride * rowv));
            return launch_pdl(tail_chain_kernel<V, long long>, blocks, stream, static_cast<V*>(mem),
                              static_cast<const V*>(hid), L, M, rowv, total, (long long)L_stride * rowv);
        }
    };
    const uintptr_t a = reinterpret_cast<uintptr_t>(mem) | reinterpret_cast<uintptr_t>(hid);
    if (row_bytes % 16 == 0 && a % 16 == 0) return go(uint4{});
    if (row_bytes % 8 == 0 && a % 8 == 0) return go(uint2{});
    if (row_bytes % 4 == 0 && a % 4 == 0) return go(uint32_t{});
    return go(uint16_t{});
}

// Ring-buffer memory (L < M): the L new rows of each batch row overwrite the
// L oldest rows of the ring, row r of h landing at ring row (start + r) mod M;
// the ring then starts at (start + L) mod M.  The logical memory (ring read
// from its start) equals the Tail_M roll of [mem; h], at the cost of writing
// L rows instead of moving M.  One thread per vector.
template <typename V, typename I>
__global__ void __launch_bounds__(256) ring_push_kernel(V* __restrict__ ring, const V* __restrict__ hid,
                                                        int L, int M, int start, I rowv, I total) {
    const I e = (I)blockIdx.x * 256 + threadIdx.x;
    if (e >= total) return;
    const I col = e % rowv;
    const I br = e / rowv;  // (b, r) of the source row
    const int r = (int)(br % (I)L);
    const I b = br / (I)L;
    int pos = start + r;
    if (pos >= M) pos -= M;
    const I ri = (b * (I)M + pos) * rowv + col;
    if (TXL_BOUNDS(pos >= 0 && pos < M && ri < (total / ((I)L * rowv)) * (I)M * rowv, 207, ri)) ring[ri] = hid[e];
}

cudaError_t launch_ring_push(void* ring, const void* hid, int B, int L, int M, int start,
                             size_t row_bytes, cudaStream_t stream) {
    auto go = [&](auto tag) -> cudaError_t {
        using V = decltype(tag);
        const long long rowv = (long long)(row_bytes / sizeof(V));
        const long long total = (long long)B * L * rowv, rsz = (long long)B * M * rowv;
        const long long blocks = (total + 255) / 256;
        if (total == 0) return cudaSuccess;
        if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
        if (rsz < 0x7FFFFFFFll - 256)
            ring_push_kernel<V, int><<<(unsigned)blocks, 256, 0, stream>>>(
                static_cast<V*>(ring), static_cast<const V*>(hid), L, M, start, (int)rowv, (int)total);
        else
            ring_push_kernel<V, long long><<<(unsigned)blocks, 256, 0, stream>>>(
                static_cast<V*>(ring), static_cast<const V*>(hid), L, M, start, rowv, total);
        return cudaGetLastError();
    };
    const uintptr_t a = reinterpret_cast<uintptr_t>(ring) | reinterpret_cast<uintptr_t>(hid);
    if (row_bytes % 16 == 0 && a % 16 == 0) return go(uint4{});
    if (row_bytes % 8 == 0 && a % 8 == 0) return go(uint2{});
    if (row_bytes % 4 == 0 && a % 4 == 0) return go(uint32_t{});
    return go(uint16_t{});
}

cudaError_t launch_mem_reset(void* mem, const unsigned char* flags, int B, long long per_b_bytes,
                             cudaStream_t stream) {
    auto go = [&](auto tag) -> cudaError_t {
        using V = decltype(tag);
        const long long per_b = per_b_bytes / (long long)sizeof(V), total = (long long)B * per_b;
        const long long blocks = (total + 255) / 256;
        if (total == 0) return cudaSuccess;
        if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
        if (total < 0x7FFFFFFFll - 256)
            mem_reset_kernel<V, int><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<V*>(mem), flags,
                                                                           (int)per_b, (int)total);
        else
            mem_reset_kernel<V, long long><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<V*>(mem), flags,
                                                                                 per_b, total);
        return cudaGetLastError();
    };
    const uintptr_t a = reinterpret_cast<uintptr_t>(mem);
    if (per_b_bytes % 16 == 0 && a % 16 == 0) return go(uint4{});
    if (per_b_bytes % 4 == 0 && a % 4 == 0) return go(uint32_t{});
    return go(uint16_t{});
}

TXL_BOUNDS_READER(bounds_word_mem_update)

}  // namespace txl
