// a4 — vocab argmax and a5 — greedy acceptance walk.
//
// The pages speak of accepted tokens and longer accepted prefixes (JETFLOW
// summary, §3 item 2 and §4) without stating a rule; the rule implemented is
// the greedy one: node i >= 1 is accepted iff its parent is accepted and its
// draft token equals the target argmax at the parent; the deepest accepted
// node wins, ties to the smallest index.
//
// argmax: a cluster of kArgCluster CTAs per logits row, each sweeping a
// contiguous slice with 16-byte loads.  Every thread keeps the first index of
// its running maximum; a batch of loaded vectors is reduced with bf16x2
// NaN-propagating max instructions and only searched for the position of its
// maximum when that maximum beats the running one, so the common path costs
// about one packed max per two logits.  The slice winners meet in CTA rank 0
// through distributed shared memory.
//
// walk: one warp per sequence.  ok[] is packed into W ballot words; node i is
// accepted iff (mask[i] & ~ok) == 0 (the root counts as ok); the best
// (depth, -index) key is found with a warp max.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace cg = cooperative_groups;

namespace tv {

constexpr int kArgThreads = 256;
constexpr int kArgCluster = 8;
constexpr int kArgBatch = 4;  // 16-byte vectors in flight per thread per batch

// (av, ai) beats (bv, bi): NaN above everything, then larger value, then smaller index.
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi)
{
    const bool an = av != av, bn = bv != bv;
    if (an != bn) return an;
    if (!an && av != bv) return av > bv;
    return ai < bi;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__global__ void __cluster_dims__(kArgCluster, 1, 1) __launch_bounds__(kArgThreads)
    argmax_kernel(const uint16_t *__restrict__ logits, long long V, long long chunk, int32_t *__restrict__ am)
{
    __shared__ float s_v[kArgThreads / 32];
    __shared__ int s_i[kArgThreads / 32];
    __shared__ float c_v;
    __shared__ int c_i;

    cg::cluster_group cluster = cg::this_cluster();
    const int part = (int)cluster.block_rank();
    const long long row_id = blockIdx.x / kArgCluster;
    const int tid = threadIdx.x;
    const uint16_t *row = logits + row_id * V;

    const long long lo = (long long)part * chunk;
    const long long hi = (lo + chunk < V) ? lo + chunk : V;

    float best_v = -__int_as_float(0x7f800000);  // -inf
    int best_i = 0x7fffffff;

    if (lo < hi) {
        // Scalar head up to the first 16-byte boundary.
        long long head = (long long)(((16u - ((uint32_t)(uintptr_t)(row + lo) & 15u)) & 15u) >> 1);
        if (head > hi - lo) head = hi - lo;
        if (tid < head) {
            const float x = bf16_bits_to_float(row[lo + tid]);
            if (beats(x, (int)(lo + tid), best_v, best_i)) { best_v = x; best_i = (int)(lo + tid); }
        }
        const long long vstart = lo + head;
        const long long nvec = (hi - vstart) / 8;
        const uint4 *vp = reinterpret_cast<const uint4 *>(row + vstart);

        for (long long base = 0; base < nvec; base += (long long)kArgThreads * kArgBatch) {
            uint4 v[kArgBatch];
            bool valid[kArgBatch];
#pragma unroll
            for (int k = 0; k < kArgBatch; ++k) {
                const long long idx = base + tid + (long long)k * kArgThreads;
                valid[k] = idx < nvec;
                v[k] = valid[k] ? __ldg(vp + idx) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
            }
            if (!valid[0]) break;
            __nv_bfloat162 m2 = *reinterpret_cast<__nv_bfloat162 *>(&v[0].x);
#pragma unroll
            for (int k = 0; k < kArgBatch; ++k) {
                m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].x));
                m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].y));
                m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].z));
                m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].w));
            }
            const float bm = __bfloat162float(__hmax_nan(m2.x, m2.y));
            const bool bm_nan = bm != bm;
            // The batch lies after everything this thread has seen, so it can only
            // win by being strictly above the running maximum (a NaN is above any
            // number; nothing is above a NaN).  Only then is it searched.
            const bool best_nan = best_v != best_v;
            const bool take = (best_i == 0x7fffffff) || (!best_nan && (bm_nan || bm > best_v));
            if (take) {
                bool found = false;
#pragma unroll
                for (int k = 0; k < kArgBatch; ++k) {
                    if (!valid[k] || found) continue;
                    const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (found) continue;
                        const float x = bf16_bits_to_float((w4[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
                        if (bm_nan ? (x != x) : (x == bm)) {
                            found = true;
                            best_v = x;
                            best_i = (int)(vstart + (base + tid + (long long)k * kArgThreads) * 8 + e);
                        }
                    }
                }
            }
        }
        // Scalar tail.
        const long long tail = vstart + nvec * 8;
        if (tid < hi - tail) {
            const float x = bf16_bits_to_float(row[tail + tid]);
            if (beats(x, (int)(tail + tid), best_v, best_i)) { best_v = x; best_i = (int)(tail + tid); }
        }
    }

    // CTA reduction.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (beats(ov, oi, best_v, best_i)) { best_v = ov; best_i = oi; }
    }
    if ((tid & 31) == 0) { s_v[tid >> 5] = best_v; s_i[tid >> 5] = best_i; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kArgThreads / 32; ++w)
            if (beats(s_v[w], s_i[w], best_v, best_i)) { best_v = s_v[w]; best_i = s_i[w]; }
        c_v = best_v;
        c_i = best_i;
    }
    // Cluster reduction in rank 0 through distributed shared memory.
    cluster.sync();
    if (part == 0 && tid == 0) {
        for (int r = 1; r < kArgCluster; ++r) {
            const float rv = *cluster.map_shared_rank(&c_v, r);
            const int ri = *cluster.map_shared_rank(&c_i, r);
            if (beats(rv, ri, best_v, best_i)) { best_v = rv; best_i = ri; }
        }
        am[row_id] = best_i;
    }
    cluster.sync();
}

constexpr int kMaxW = 8;

__global__ void __launch_bounds__(32) accept_walk_kernel(const int32_t *__restrict__ am,
                                                         const int32_t *__restrict__ draft,
                                                         const int32_t *__restrict__ parent,
                                                         const uint32_t *__restrict__ mask, int B, int W,
                                                         int32_t *__restrict__ n_acc, int32_t *__restrict__ path,
                                                         int32_t *__restrict__ bonus, int32_t *status)
{
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    const int32_t *amb = am + (size_t)b * B;
    bool bad = false;

    uint32_t okw[kMaxW];
#pragma unroll
    for (int k = 0; k < kMaxW; ++k) {
        const int node = k * 32 + lane;
        bool ok = true;
        if (k < W && node > 0 && node < B) {
            const int p = parent[(size_t)b * B + node];
            if (p < 0 || p >= node) {
                bad = true;
                ok = false;
            } else {
                ok = draft[(size_t)b * B + node] == amb[p];
            }
        }
        okw[k] = __ballot_sync(0xffffffffu, ok);
    }

    int best = -1;  // key = depth * 512 + (511 - node)
#pragma unroll
    for (int k = 0; k < kMaxW; ++k) {
        const int node = k * 32 + lane;
        if (k < W && node < B) {
            const uint32_t *mrow = mask + ((size_t)b * B + node) * W;
            bool acc = true;
            int bits = 0;
#pragma unroll
            for (int w = 0; w < kMaxW; ++w) {
                if (w < W) {
                    const uint32_t mw = mrow[w];
                    acc = acc && ((mw & ~okw[w]) == 0u);
                    bits += __popc(mw);
                }
            }
            if (acc) best = max(best, (bits - 1) * 512 + (511 - node));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
    bad = __any_sync(0xffffffffu, bad);

    const int vstar = (best >= 0) ? 511 - (best & 511) : 0;
    const int dep = (best >= 0) ? (best >> 9) : 0;
    const uint32_t *vrow = mask + ((size_t)b * B + vstar) * W;
    int before = 0;
#pragma unroll
    for (int k = 0; k < kMaxW; ++k) {
        if (k < W) {
            const uint32_t mw = vrow[k];
            const int node = k * 32 + lane;
            if ((mw >> lane) & 1u) path[(size_t)b * B + before + __popc(mw & ((1u << lane) - 1u))] = node;
            before += __popc(mw);
            if (node < B && node > dep) path[(size_t)b * B + node] = -1;
        }
    }
    if (lane == 0) {
        n_acc[b] = dep;
        bonus[b] = amb[vstar];
        if (bad) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
    }
}

cudaError_t launch_accept(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                          const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                          int32_t *bonus, int32_t *status, cudaStream_t stream)
{
    const long long rows = (long long)nb * B;
    long long chunk = ((long long)V + kArgCluster - 1) / kArgCluster;
    chunk = (chunk + 7) / 8 * 8;
    argmax_kernel<<<(unsigned)(rows * kArgCluster), kArgThreads, 0, stream>>>(logits, V, chunk, am);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int W = (B + 31) / 32;
    accept_walk_kernel<<<nb, 32, 0, stream>>>(am, draft, parent, mask, B, W, n_acc, path, bonus, status);
    return cudaGetLastError();
}

}  // namespace tv
