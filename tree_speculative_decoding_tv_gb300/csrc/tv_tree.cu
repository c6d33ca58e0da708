// Best-first draft-tree construction with top-w rounds.
//
// JETFLOW summary, §2 "Estrategia de Entrenamiento": the draft head emits logits
// for every tree depth at once; a branch score (by default the cumulative draft
// log-probability) ranks the nodes and best-first expansion builds the tree up to
// a budget.  DFlash-TfM summary, §2 "Construcción de Árboles": the top w
// candidates of the heap are expanded together, so B nodes take ceil(B/w) rounds.
// Depth d's candidates are K (token, log-prob) pairs sorted best first, the same
// for every node at depth d-1; a candidate child (u, c) scores score[u] +
// logp[d][c] in fp32; ties go to the smaller parent index, then the smaller rank.
//
// GPU form: one warp per sequence.  Because each depth's log-probs are sorted,
// a node's best remaining candidate is always its next rank, so the frontier
// holds one entry per node (its next child) instead of all K: at most B entries,
// kept in registers (9 slots per lane).  Each lane keeps the best of its own
// slots; a pop is a warp max of the order-preserving score followed by a warp min
// of (parent, rank) among the lanes holding it (two single-instruction
// reductions), and only the lane owning a changed slot looks again.  The popped
// entry's sibling successor joins the frontier at once (it was a candidate when
// the round began); the round's new nodes add their first children only when the
// round ends, which is what expanding the w nodes together means.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kTreeMaxB = 256;
constexpr int kTreeSlots = 9;  // frontier slots per lane: 9 x 32 >= kTreeMaxB

// Order-preserving image of a finite score (larger score -> larger value, never 0).
__device__ __forceinline__ uint32_t score_key(float s)
{
    const uint32_t b = __float_as_uint(s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr int kTreeSmemLp = 8192;  // log-prob tables up to this size are staged in shared memory

__global__ void __launch_bounds__(32) build_tree_kernel(const float *__restrict__ logp, const int32_t *__restrict__ tok,
                                                        int Dmax, int K, int B, int w, int32_t *__restrict__ parent,
                                                        int32_t *__restrict__ token, float *__restrict__ score,
                                                        int32_t *status)
{
    __shared__ float sc[kTreeMaxB];
    __shared__ int16_t dep[kTreeMaxB], par[kTreeMaxB], rank[kTreeMaxB];
    __shared__ float s_lp[kTreeSmemLp];
    const int b = blockIdx.x, lane = threadIdx.x;
    const float *g_lp = logp + (size_t)b * Dmax * K;
    const int32_t *tk = tok + (size_t)b * Dmax * K;

    pdl_wait_primary();
    pdl_launch_dependents();
    // each depth's log-probs finite and sorted best first; small tables go to shared memory
    const bool staged = Dmax * K <= kTreeSmemLp;
    bool bad = false;
    for (int t = lane; t < Dmax * K; t += 32) {
        const float x = g_lp[t];
        if (!(fabsf(x) <= 3.0e38f)) bad = true;
        if (t % K + 1 < K && !(x >= g_lp[t + 1])) bad = true;
        if (staged) s_lp[t] = x;
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) report_status(status, TV_ERR_INVALID_ARG);
        return;
    }
    const float *lp = staged ? s_lp : g_lp;

    // The frontier lives in registers: slot j is register q = j / 32 of lane j % 32.
    // rt = (parent << 16) | rank, or kEmpty; rf = the candidate's score.  Slots are
    // never compacted: a parent whose ranks run out leaves an empty slot behind.
    constexpr uint32_t kEmpty = 0xFFFFFFFFu;
    float rf[kTreeSlots];
    uint32_t rt[kTreeSlots];
#pragma unroll
    for (int q = 0; q < kTreeSlots; ++q) {
        rf[q] = 0.f;
        rt[q] = kEmpty;
    }
    uint32_t my_s = 0, my_t = kEmpty;  // this lane's best slot: score key, tie-break, score, register
    float my_f = 0.f;
    int my_q = 0;
    auto lane_best = [&]() {
        my_s = 0;
        my_t = kEmpty;
#pragma unroll
        for (int q = 0; q < kTreeSlots; ++q) {
            if (rt[q] != kEmpty) {
                const uint32_t k = score_key(rf[q]);
                if (k > my_s || (k == my_s && rt[q] < my_t)) {
                    my_s = k;
                    my_t = rt[q];
                    my_f = rf[q];
                    my_q = q;
                }
            }
        }
    };
    // slot j <- (f, t), by its owner lane
    auto put = [&](int j, float f, uint32_t t) {
        if ((j & 31) == lane) {
            const int qj = j >> 5;
#pragma unroll
            for (int q = 0; q < kTreeSlots; ++q)
                if (q == qj) {
                    rf[q] = f;
                    rt[q] = t;
                }
            lane_best();
        }
    };

    if (lane == 0) {
        sc[0] = 0.f;
        dep[0] = 0;
        par[0] = -1;
        rank[0] = 0;
    }
    int n = 1, made = 1;  // slots used, nodes made (warp-uniform)
    put(0, 0.f + lp[0], 0u);
    __syncwarp();
    while (made < B) {
        const int take = min(w, B - made);
        const int first = made;
        for (int t = 0; t < take; ++t) {
            // the best entry: largest score key, then smallest (parent, rank)
            const uint32_t top_s = __reduce_max_sync(0xffffffffu, my_s);
            if (top_s == 0) break;  // no candidate left this round
            const uint32_t top_t = __reduce_min_sync(0xffffffffu, my_s == top_s ? my_t : kEmpty);
            const int owner = __ffs(__ballot_sync(0xffffffffu, my_s == top_s && my_t == top_t)) - 1;
            const float f = __shfl_sync(0xffffffffu, my_f, owner);
            const int u = (int)(top_t >> 16), c = (int)(top_t & 0xFFFFu), i = made;
            const int d = dep[u] + 1;
            if (lane == 0) {
                par[i] = (int16_t)u;
                dep[i] = (int16_t)d;
                rank[i] = (int16_t)c;
                sc[i] = f;
            }
            // the parent's next rank takes the popped slot, or the slot empties
            if (lane == owner) {
                const int q = my_q;
                const bool more = c + 1 < K;
                const float nf = more ? sc[u] + lp[(size_t)(d - 1) * K + c + 1] : 0.f;
#pragma unroll
                for (int qq = 0; qq < kTreeSlots; ++qq)
                    if (qq == q) {
                        rf[qq] = nf;
                        rt[qq] = more ? (((uint32_t)u << 16) | (uint32_t)(c + 1)) : kEmpty;
                    }
                lane_best();
            }
            ++made;
            __syncwarp();
        }
        // the round's nodes join with their first child
        for (int i = first; i < made; ++i) {
            const int di = dep[i];
            if (di < Dmax) {
                put(n, sc[i] + lp[(size_t)di * K], (uint32_t)i << 16);
                ++n;
            }
        }
        __syncwarp();
        if (__reduce_max_sync(0xffffffffu, my_s) == 0) break;  // no candidate at all: B exceeds the tree
    }
    if (made < B && lane == 0) report_status(status, TV_ERR_INVALID_ARG);
    for (int i = lane; i < B; i += 32) {
        const bool ok = i < made;
        parent[(size_t)b * B + i] = ok ? par[i] : -1;
        token[(size_t)b * B + i] = (ok && i > 0) ? tk[(size_t)(dep[i] - 1) * K + rank[i]] : -1;
        score[(size_t)b * B + i] = ok ? sc[i] : 0.f;
    }
}

cudaError_t launch_build_tree(const float *logp, const int32_t *tok, int nb, int Dmax, int K, int B, int w,
                              int32_t *parent, int32_t *token, float *score, int32_t *status, cudaStream_t stream)
{
    return launch_dependent(build_tree_kernel, dim3((unsigned)nb), dim3(32), 0, stream, logp, tok, Dmax, K, B, w,
                            parent, token, score, status);
}

}  // namespace tv
