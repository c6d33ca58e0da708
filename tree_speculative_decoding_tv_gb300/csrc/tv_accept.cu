// a4 — vocab argmax and a5 — greedy acceptance walk.
//
// The pages speak of accepted tokens and longer accepted prefixes (JETFLOW
// summary, §3 item 2 and §4) without stating a rule; the rule implemented is
// the greedy one: node i >= 1 is accepted iff its parent is accepted and its
// draft token equals the target argmax at the parent; the deepest accepted
// node wins, ties to the smallest index.
//
// argmax (kernel 1): the logits are cut into (row, 8192-element chunk) units
// and a one-wave grid walks them, so every SM streams the same number of
// bytes whatever the row count.  A unit is one 16-byte-vector batch per
// thread: bf16x2 NaN-propagating max instructions reduce it (about one per two
// logits), the CTA agrees on the unit's maximum, and only the threads that
// hold it search for its first position.  One (value, index) partial per unit
// goes to the caller's workspace.
//
// accept (kernel 2): one CTA per sequence, one thread per node.  Each thread
// finishes its row's argmax from the chunk partials, then ok[] is packed into
// W ballot words; node i is accepted iff (mask[i] & ~ok) == 0 (the root counts
// as ok); the best (depth, -index) key is a block max; the path is read off
// the chosen node's mask bits in ascending order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kArgThreads = 256;
constexpr int kArgChunk = 8192;   // logits per unit (16 KB)
constexpr int kArgBatch = 4;      // 16-byte vectors per thread per batch
constexpr int kArgCtasPerSm = 8;
constexpr int kMaxB = 256;
constexpr int kMaxW = kMaxB / 32;

// (av, ai) beats (bv, bi): NaN above everything, then larger value, then smaller index.
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi)
{
    const bool an = av != av, bn = bv != bv;
    if (an != bn) return an;
    if (!an && av != bv) return av > bv;
    return ai < bi;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ unsigned long long pack_best(float v, int i)
{
    return ((unsigned long long)(uint32_t)i << 32) | __float_as_uint(v);
}

// max with a NaN counting as the largest value
__device__ __forceinline__ float max_nan(float a, float b) { return (a != a) ? a : ((b != b) ? b : fmaxf(a, b)); }

// One unit = one batch: every thread holds its kArgBatch vectors in registers,
// the CTA first agrees on the unit's maximum value, and only the threads that
// hold that value look for its first position.
__global__ void __launch_bounds__(kArgThreads) argmax_partial_kernel(const uint16_t *__restrict__ logits, long long V,
                                                                     int nchunk, long long units,
                                                                     unsigned long long *__restrict__ part)
{
    static_assert(kArgChunk == kArgThreads * kArgBatch * 8, "one batch per unit");
    __shared__ float s_v[kArgThreads / 32];
    __shared__ int s_i[kArgThreads / 32];
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;
    const float NEG_INF = -__int_as_float(0x7f800000);

    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const long long row_id = u / nchunk;
        const long long lo = (u - row_id * nchunk) * (long long)kArgChunk;
        const long long hi = (lo + kArgChunk < V) ? lo + kArgChunk : V;
        const uint16_t *row = logits + row_id * V;

        // scalar head up to the first 16-byte boundary, 16-byte vectors, scalar tail
        long long head = (long long)(((16u - ((uint32_t)(uintptr_t)(row + lo) & 15u)) & 15u) >> 1);
        if (head > hi - lo) head = hi - lo;
        const long long vstart = lo + head;
        const long long nvec = (hi - vstart) / 8;
        const long long tail = vstart + nvec * 8;
        const uint4 *vp = reinterpret_cast<const uint4 *>(row + vstart);
        uint4 v[kArgBatch];
        bool valid[kArgBatch];
#pragma unroll
        for (int k = 0; k < kArgBatch; ++k) {
            const long long idx = tid + (long long)k * kArgThreads;
            valid[k] = idx < nvec;
            v[k] = valid[k] ? __ldcs(vp + idx) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
        const bool has_head = tid < head, has_tail = tid < hi - tail;
        const float xh = has_head ? bf16_bits_to_float(row[lo + tid]) : NEG_INF;
        const float xt = has_tail ? bf16_bits_to_float(row[tail + tid]) : NEG_INF;

        __nv_bfloat162 m2 = *reinterpret_cast<__nv_bfloat162 *>(&v[0].x);
#pragma unroll
        for (int k = 0; k < kArgBatch; ++k) {
            m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].x));
            m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].y));
            m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].z));
            m2 = __hmax2_nan(m2, *reinterpret_cast<__nv_bfloat162 *>(&v[k].w));
        }
        float tm = max_nan(max_nan(__bfloat162float(__hmax_nan(m2.x, m2.y)), xh), xt);

        // the unit's maximum value
        float bm = tm;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bm = max_nan(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        if (lane == 0) s_v[wid] = bm;
        __syncthreads();
        bm = s_v[0];
#pragma unroll
        for (int w = 1; w < kArgThreads / 32; ++w) bm = max_nan(bm, s_v[w]);
        const bool bm_nan = bm != bm;

        // the first position holding it (elements in index order: head, vectors, tail)
        int idx = 0x7fffffff;
        if (bm_nan ? (tm != tm) : (tm == bm)) {
            if (has_head && (bm_nan ? (xh != xh) : (xh == bm))) idx = (int)(lo + tid);
#pragma unroll
            for (int k = 0; k < kArgBatch; ++k) {
                const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = bf16_bits_to_float((w4[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
                    const int pos = (int)(vstart + (tid + (long long)k * kArgThreads) * 8 + e);
                    if (valid[k] && (bm_nan ? (x != x) : (x == bm))) idx = min(idx, pos);
                }
            }
            if (has_tail && (bm_nan ? (xt != xt) : (xt == bm))) idx = min(idx, (int)(tail + tid));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
        if (lane == 0) s_i[wid] = idx;
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int w = 1; w < kArgThreads / 32; ++w) idx = min(idx, s_i[w]);
            part[u] = pack_best(bm, idx);
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kMaxB) accept_kernel(const unsigned long long *__restrict__ part, int nchunk,
                                                       const int32_t *__restrict__ draft,
                                                       const int32_t *__restrict__ parent,
                                                       const uint32_t *__restrict__ mask, int B, int W,
                                                       int32_t *__restrict__ am, int32_t *__restrict__ n_acc,
                                                       int32_t *__restrict__ path, int32_t *__restrict__ bonus,
                                                       int32_t *status)
{
    __shared__ int s_am[kMaxB];
    __shared__ uint32_t s_ok[kMaxW];
    __shared__ uint32_t s_vmask[kMaxW];
    __shared__ int s_best[kMaxB / 32];
    __shared__ int s_bad;

    const int b = blockIdx.x;
    const int i = threadIdx.x;
    const int lane = i & 31, wid = i >> 5;
    if (i == 0) s_bad = 0;

    // finish the argmax of row (b, i) from its chunk partials
    if (i < B) {
        const unsigned long long *pr = part + ((size_t)b * B + i) * nchunk;
        unsigned long long pk = pr[0];
        float bv = __uint_as_float((uint32_t)pk);
        int bi = (int)(pk >> 32);
        for (int c = 1; c < nchunk; ++c) {
            pk = pr[c];
            const float v = __uint_as_float((uint32_t)pk);
            const int ix = (int)(pk >> 32);
            if (beats(v, ix, bv, bi)) {
                bv = v;
                bi = ix;
            }
        }
        s_am[i] = bi;
        am[(size_t)b * B + i] = bi;
    }
    __syncthreads();

    bool ok = true;
    if (i > 0 && i < B) {
        const int p = parent[(size_t)b * B + i];
        if (p < 0 || p >= i) {
            ok = false;
            s_bad = 1;
        } else {
            ok = draft[(size_t)b * B + i] == s_am[p];
        }
    }
    const uint32_t okw = __ballot_sync(0xffffffffu, ok);
    if (lane == 0 && wid < kMaxW) s_ok[wid] = okw;
    __syncthreads();

    int key = -1;  // depth * 512 + (511 - node) of an accepted node
    if (i < B) {
        const uint32_t *mrow = mask + ((size_t)b * B + i) * W;
        bool acc = true;
        int bits = 0;
        for (int w = 0; w < W; ++w) {
            const uint32_t mw = mrow[w];
            acc = acc && ((mw & ~s_ok[w]) == 0u);
            bits += __popc(mw);
        }
        if (acc) key = (bits - 1) * 512 + (511 - i);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    if (lane == 0) s_best[wid] = key;
    __syncthreads();
    if (i == 0) {
        int k = s_best[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) k = max(k, s_best[w]);
        s_best[0] = k;
    }
    __syncthreads();
    const int best = s_best[0];
    const int vstar = best >= 0 ? 511 - (best & 511) : 0;
    const int dep = best >= 0 ? (best >> 9) : 0;
    if (i < W) s_vmask[i] = mask[((size_t)b * B + vstar) * W + i];
    __syncthreads();

    if (i < B) {
        const int w = i >> 5;
        const uint32_t mw = s_vmask[w];
        if ((mw >> lane) & 1u) {
            int before = __popc(mw & ((1u << lane) - 1u));
            for (int k = 0; k < w; ++k) before += __popc(s_vmask[k]);
            path[(size_t)b * B + before] = i;
        }
        if (i > dep) path[(size_t)b * B + i] = -1;
    }
    if (i == 0) {
        n_acc[b] = dep;
        bonus[b] = s_am[vstar];
        if (s_bad) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
    }
}

size_t accept_workspace_bytes(int V, int B, int nb)
{
    const long long nchunk = ((long long)V + kArgChunk - 1) / kArgChunk;
    return (size_t)nb * B * nchunk * sizeof(unsigned long long);
}

cudaError_t launch_accept(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                          const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                          int32_t *bonus, int32_t *status, void *workspace, int num_sms, cudaStream_t stream)
{
    const int nchunk = (int)(((long long)V + kArgChunk - 1) / kArgChunk);
    const long long units = (long long)nb * B * nchunk;
    long long grid = (long long)num_sms * kArgCtasPerSm;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    unsigned long long *part = static_cast<unsigned long long *>(workspace);
    argmax_partial_kernel<<<(unsigned)grid, kArgThreads, 0, stream>>>(logits, V, nchunk, units, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int W = (B + 31) / 32;
    const int threads = ((B + 31) / 32) * 32;
    accept_kernel<<<nb, threads, 0, stream>>>(part, nchunk, draft, parent, mask, B, W, am, n_acc, path, bonus,
                                              status);
    return cudaGetLastError();
}

}  // namespace tv
