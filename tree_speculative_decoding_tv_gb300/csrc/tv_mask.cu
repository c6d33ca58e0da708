// Packed ancestor masks and depths of a topologically ordered draft tree.
//
// Definition (JETFLOW summary, §2 "Arquitectura Central", tree-causal mask;
// DFlash-TfM summary, §3 "Solución", topological order): node i may attend to
// itself and to its ancestors, anc[0] = {0}, anc[i] = anc[parent[i]] U {i}.
//
// GPU form: one CTA per sequence, one thread per node, pointer doubling in
// shared memory.  After round k every node holds its ancestors at distance
// < 2^k and a pointer to its 2^k-th ancestor, so ceil(log2(depth + 1)) rounds
// of row ORs (16-byte vectors for wide rows) replace a depth-long sequential
// walk; the rounds stop as soon as no node has an ancestor left to jump to.
#include <cuda_runtime.h>

#include <type_traits>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kMaskMaxB = 256;
constexpr int kMaskMaxW = kMaskMaxB / 32;

// The rows of one buffer, WP (a power of two >= W) words each; WP >= 4 moves a
// row as 16-byte vectors.
template <int WP>
struct MaskRows {
    static constexpr int kVec = WP >= 4 ? WP / 4 : 1;
    using T = typename std::conditional<WP >= 4, uint4, typename std::conditional<WP == 2, uint2, uint32_t>::type>::type;
    T v[kMaskMaxB][kVec];
};

__device__ __forceinline__ uint32_t or_words(uint32_t a, uint32_t b) { return a | b; }
__device__ __forceinline__ uint2 or_words(uint2 a, uint2 b) { return make_uint2(a.x | b.x, a.y | b.y); }
__device__ __forceinline__ uint4 or_words(uint4 a, uint4 b) { return make_uint4(a.x | b.x, a.y | b.y, a.z | b.z, a.w | b.w); }

template <int WP>
__global__ void __launch_bounds__(kMaskMaxB) build_mask_kernel(const int32_t *__restrict__ parent, int B, int W,
                                                               uint32_t *__restrict__ mask, int32_t *__restrict__ depth,
                                                               int32_t *status)
{
    using R = MaskRows<WP>;
    constexpr int kVec = R::kVec;
    __shared__ __align__(16) R anc[2];
    __shared__ int16_t jump[2][kMaskMaxB];

    const int b = blockIdx.x;
    const int i = threadIdx.x;
    pdl_wait_primary();        // parent[] may come from the previous kernel in the stream
    pdl_launch_dependents();   // the attention kernel may start its set-up meanwhile

    int p = -1;
    bool ok = true;
    if (i < B) {
        p = parent[(size_t)b * B + i];
        ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
        if (!ok) p = -1;  // keep the doubling in bounds; the status word reports the error
    }
    uint32_t *own = reinterpret_cast<uint32_t *>(&anc[0].v[i][0]);
#pragma unroll
    for (int w = 0; w < kVec * (sizeof(typename R::T) / 4); ++w)
        own[w] = (i < B && w == (i >> 5)) ? (1u << (i & 31)) : 0u;
    jump[0][i] = (int16_t)p;
    const bool bad = __syncthreads_or(!ok);

    // Doubling: after a round every node holds its ancestors at distance < 2^k and
    // its 2^k-th ancestor.  Once no node has an ancestor left to jump to, every
    // set is complete, so the rounds stop at ceil(log2(depth + 1)).
    int cur = 0;
    for (;;) {
        const int j = jump[cur][i];
        if (!__syncthreads_or(j >= 0)) break;  // also orders the previous round's writes
        const int nxt = cur ^ 1;
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
            const typename R::T mine = anc[cur].v[i][q];
            anc[nxt].v[i][q] = (j >= 0) ? or_words(mine, anc[cur].v[j][q]) : mine;
        }
        jump[nxt][i] = (j >= 0) ? jump[cur][j] : (int16_t)-1;
        cur = nxt;
    }

    // coalesced stores of the sequence's B x W words; depth = ancestor count - 1
    const uint32_t *rows = reinterpret_cast<const uint32_t *>(&anc[cur].v[0][0]);
    constexpr int kStride = kVec * (sizeof(typename R::T) / 4);
    uint32_t *out = mask + (size_t)b * B * W;
    for (int t = i; t < B * W; t += blockDim.x) {
        const int r = t / W, w = t - r * W;
        out[t] = rows[r * kStride + w];
    }
    if (i < B && depth) {
        int bits = 0;
#pragma unroll
        for (int w = 0; w < kStride; ++w) bits += __popc(rows[i * kStride + w]);
        depth[(size_t)b * B + i] = bits - 1;
    }
    if (i == 0 && bad) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
}

cudaError_t launch_build_mask(const int32_t *parent, int B, int nb, uint32_t *mask, int32_t *depth, int32_t *status,
                              cudaStream_t stream)
{
    const int W = (B + 31) / 32;
    const int threads = W * 32;
    if (W == 1)
        return launch_dependent(build_mask_kernel<1>, dim3(nb), dim3(threads), 0, stream, parent, B, W, mask, depth, status);
    if (W == 2)
        return launch_dependent(build_mask_kernel<2>, dim3(nb), dim3(threads), 0, stream, parent, B, W, mask, depth, status);
    if (W <= 4)
        return launch_dependent(build_mask_kernel<4>, dim3(nb), dim3(threads), 0, stream, parent, B, W, mask, depth, status);
    return launch_dependent(build_mask_kernel<8>, dim3(nb), dim3(threads), 0, stream, parent, B, W, mask, depth, status);
}

}  // namespace tv
