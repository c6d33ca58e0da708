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
// round ends, which is what expanding the w nodes together means.  Each slot keeps
// its parent's score and its depth in registers, and each lane prepares its best
// slot's successor before the reductions; a lane's best is a 64-bit max over its
// slots (a tournament after a pop, one comparison after an insertion), so a pop's
// dependent chain is the two reductions, a shuffle and a few register operations.
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
    // rt = (parent << 16) | rank, or kEmpty; rf = the candidate's score; rp = its
    // parent's score; rd = its depth.  Slots are never compacted: a parent whose
    // ranks run out leaves an empty slot behind.
    constexpr uint32_t kEmpty = 0xFFFFFFFFu;
    float rf[kTreeSlots], rp[kTreeSlots];
    uint32_t rt[kTreeSlots];
    int rd[kTreeSlots];
#pragma unroll
    for (int q = 0; q < kTreeSlots; ++q) {
        rf[q] = rp[q] = 0.f;
        rt[q] = kEmpty;
        rd[q] = 0;
    }
    // this lane's best slot (score key, tie-break, score, depth) and, ready before the
    // pop that may take it, that slot's replacement: the parent's next rank.  A slot's
    // order is one 64-bit value, (score key << 32) | ~tie-break (0 for an empty slot),
    // so the best is a max over the slots.
    uint32_t my_s = 0, my_t = kEmpty, rep_t = kEmpty;
    float my_f = 0.f, my_p = 0.f, rep_f = 0.f;
    int my_d = 0;
    auto order = [&](float f, uint32_t t) -> uint64_t {
        return t == kEmpty ? 0ull : (((uint64_t)score_key(f) << 32) | (uint64_t)(~t));
    };
    auto prepare = [&]() {  // the replacement of the best slot
        const int c = (int)(my_t & 0xFFFFu);
        if (my_t != kEmpty && c + 1 < K) {
            rep_f = my_p + lp[(size_t)(my_d - 1) * K + c + 1];
            rep_t = my_t + 1u;
        } else {
            rep_t = kEmpty;
        }
    };
    auto lane_best = [&]() {  // full rescan: a tournament over the slots
        uint64_t o[kTreeSlots];
#pragma unroll
        for (int q = 0; q < kTreeSlots; ++q) o[q] = order(rf[q], rt[q]);
#pragma unroll
        for (int step = 1; step < kTreeSlots; step <<= 1)
#pragma unroll
            for (int q = 0; q + step < kTreeSlots; q += 2 * step) o[q] = o[q] > o[q + step] ? o[q] : o[q + step];
        my_s = (uint32_t)(o[0] >> 32);
        my_t = ~(uint32_t)o[0];
        if (o[0] == 0ull) my_t = kEmpty;
#pragma unroll
        for (int q = 0; q < kTreeSlots; ++q)
            if (rt[q] == my_t && my_t != kEmpty) {
                my_f = rf[q];
                my_p = rp[q];
                my_d = rd[q];
            }
        prepare();
    };
    // slot j <- a candidate (score f, tie-break t) with parent score ps at depth d, by its
    // owner lane; the lane's best changes only if the newcomer beats it
    auto put = [&](int j, float f, uint32_t t, float ps, int d) {
        if ((j & 31) == lane) {
            const int qj = j >> 5;
#pragma unroll
            for (int q = 0; q < kTreeSlots; ++q)
                if (q == qj) {
                    rf[q] = f;
                    rt[q] = t;
                    rp[q] = ps;
                    rd[q] = d;
                }
            if (order(f, t) > order(my_f, my_t)) {
                my_s = score_key(f);
                my_t = t;
                my_f = f;
                my_p = ps;
                my_d = d;
                prepare();
            }
        }
    };

    if (lane == 0) {
        sc[0] = 0.f;
        dep[0] = 0;
        par[0] = -1;
        rank[0] = 0;
    }
    int n = 1, made = 1;  // slots used, nodes made (warp-uniform)
    put(0, 0.f + lp[0], 0u, 0.f, 1);
    __syncwarp();
    float last_f = 0.f;  // the last popped node's score and depth (the w = 1 round's only node)
    int last_d = 0;
    // w = 1: every round is one pop, after which the popped node's first child joins.  Both
    // frontier updates (the popped slot's replacement by its owner lane, the child's slot by
    // its lane) go in one pass; a lane doing both rescans once, over the same slots the two
    // steps would compare.  A top score that one lane alone holds needs no second reduction.
    while (w == 1 && made < B) {
        const uint32_t top_s = __reduce_max_sync(0xffffffffu, my_s);
        if (top_s == 0) break;  // no candidate left: B exceeds the tree
        const unsigned hold = __ballot_sync(0xffffffffu, my_s == top_s);
        int owner;
        uint32_t top_t;
        if (__popc(hold) == 1) {
            owner = __ffs(hold) - 1;
            top_t = __shfl_sync(0xffffffffu, my_t, owner);
        } else {
            top_t = __reduce_min_sync(0xffffffffu, my_s == top_s ? my_t : kEmpty);
            owner = __ffs(__ballot_sync(0xffffffffu, my_s == top_s && my_t == top_t)) - 1;
        }
        const float f = __shfl_sync(0xffffffffu, my_f, owner);
        const int d = __shfl_sync(0xffffffffu, my_d, owner);
        const int i = made;
        if (lane == 0) {
            par[i] = (int16_t)(top_t >> 16);
            dep[i] = (int16_t)d;
            rank[i] = (int16_t)(top_t & 0xFFFFu);
            sc[i] = f;
        }
        const bool child = d < Dmax;  // node i's first child: slot n, parent score f, depth d + 1
        const float cf = child ? f + lp[(size_t)d * K] : 0.f;
        const uint32_t ct = (uint32_t)i << 16;
        const bool ins = child && (n & 31) == lane, own = lane == owner;
        if (own) {
#pragma unroll
            for (int q = 0; q < kTreeSlots; ++q)
                if (rt[q] == top_t) {
                    rf[q] = rep_f;
                    rt[q] = rep_t;
                }
        }
        if (ins) {
            const int qn = n >> 5;
#pragma unroll
            for (int q = 0; q < kTreeSlots; ++q)
                if (q == qn) {
                    rf[q] = cf;
                    rt[q] = ct;
                    rp[q] = f;
                    rd[q] = d + 1;
                }
        }
        if (own) {
            lane_best();
        } else if (ins && order(cf, ct) > order(my_f, my_t)) {
            my_s = score_key(cf);
            my_t = ct;
            my_f = cf;
            my_p = f;
            my_d = d + 1;
            prepare();
        }
        if (child) ++n;
        ++made;
        __syncwarp();
    }
    while (w != 1 && made < B) {
        const int take = min(w, B - made);
        const int first = made;
        for (int t = 0; t < take; ++t) {
            // the best entry: largest score key, then smallest (parent, rank)
            const uint32_t top_s = __reduce_max_sync(0xffffffffu, my_s);
            if (top_s == 0) break;  // no candidate left this round
            const uint32_t top_t = __reduce_min_sync(0xffffffffu, my_s == top_s ? my_t : kEmpty);
            const int owner = __ffs(__ballot_sync(0xffffffffu, my_s == top_s && my_t == top_t)) - 1;
            const float f = __shfl_sync(0xffffffffu, my_f, owner);
            const int d = __shfl_sync(0xffffffffu, my_d, owner);
            const int u = (int)(top_t >> 16), c = (int)(top_t & 0xFFFFu), i = made;
            if (lane == 0) {
                par[i] = (int16_t)u;
                dep[i] = (int16_t)d;
                rank[i] = (int16_t)c;
                sc[i] = f;
            }
            // the parent's next rank (computed ahead) takes the popped slot, or the slot empties
            if (lane == owner) {
#pragma unroll
                for (int q = 0; q < kTreeSlots; ++q)
                    if (rt[q] == top_t) {
                        rf[q] = rep_f;
                        rt[q] = rep_t;
                    }
                lane_best();
            }
            last_f = f;
            last_d = d;
            ++made;
            __syncwarp();
        }
        // the round's nodes join with their first child
        for (int i = first; i < made; ++i) {
            const bool lastn = i == made - 1;
            const float fi = lastn ? last_f : sc[i];
            const int di = lastn ? last_d : dep[i];
            if (di < Dmax) {
                put(n, fi + lp[(size_t)di * K], (uint32_t)i << 16, fi, di + 1);
                ++n;
            }
        }
        __syncwarp();
        if (made == first) break;  // the round found no candidate at all: B exceeds the tree
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
