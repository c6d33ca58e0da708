// a1 — packed ancestor masks and depths of a topologically ordered draft tree.
//
// Definition (JETFLOW summary, §2 "Arquitectura Central", tree-causal mask;
// DFlash-TfM summary, §3 "Solución", topological order): node i may attend to
// itself and to its ancestors, anc[0] = {0}, anc[i] = anc[parent[i]] U {i}.
//
// GPU form: one CTA per sequence, one thread per node, pointer doubling in
// shared memory.  After round k every node holds its ancestors at distance
// < 2^k and a pointer to its 2^k-th ancestor, so ceil(log2 B) rounds of W-word
// ORs replace a depth-long sequential walk.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kMaskMaxB = 256;
constexpr int kMaskMaxW = kMaskMaxB / 32;

__global__ void __launch_bounds__(kMaskMaxB) build_mask_kernel(const int32_t *__restrict__ parent, int B, int W,
                                                               uint32_t *__restrict__ mask, int32_t *__restrict__ depth,
                                                               int32_t *status)
{
    __shared__ uint32_t anc[2][kMaskMaxB][kMaskMaxW];
    __shared__ int16_t jump[2][kMaskMaxB];
    __shared__ int bad;

    const int b = blockIdx.x;
    const int i = threadIdx.x;
    if (i == 0) bad = 0;
    pdl_wait_primary();        // parent[] may come from the previous kernel in the stream
    pdl_launch_dependents();   // the attention kernel may start its set-up meanwhile
    __syncthreads();

    int p = -1;
    if (i < B) {
        p = parent[(size_t)b * B + i];
        const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
        if (!ok) {
            bad = 1;
            p = -1;  // keep the doubling in bounds; the status word reports the error
        }
    }
    for (int w = 0; w < W; ++w) anc[0][i][w] = (i < B && w == (i >> 5)) ? (1u << (i & 31)) : 0u;
    jump[0][i] = (int16_t)p;
    __syncthreads();

    const int rounds = (B > 1) ? 32 - __clz(B - 1) : 0;
    int cur = 0;
    for (int k = 0; k < rounds; ++k) {
        const int j = jump[cur][i];
        for (int w = 0; w < W; ++w) anc[cur ^ 1][i][w] = anc[cur][i][w] | (j >= 0 ? anc[cur][j][w] : 0u);
        jump[cur ^ 1][i] = (j >= 0) ? jump[cur][j] : (int16_t)-1;
        __syncthreads();
        cur ^= 1;
    }

    if (i < B) {
        uint32_t *row = mask + ((size_t)b * B + i) * W;
        int bits = 0;
        for (int w = 0; w < W; ++w) {
            row[w] = anc[cur][i][w];
            bits += __popc(anc[cur][i][w]);
        }
        if (depth) depth[(size_t)b * B + i] = bits - 1;
    }
    if (i == 0 && bad) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
}

cudaError_t launch_build_mask(const int32_t *parent, int B, int nb, uint32_t *mask, int32_t *depth, int32_t *status,
                              cudaStream_t stream)
{
    const int W = (B + 31) / 32;
    const int threads = ((B + 31) / 32) * 32;
    return launch_dependent(build_mask_kernel, dim3(nb), dim3(threads), 0, stream, parent, B, W, mask, depth, status);
}

}  // namespace tv
