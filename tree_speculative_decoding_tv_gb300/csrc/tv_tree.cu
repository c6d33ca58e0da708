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
// GPU form: one CTA of 256 threads per sequence, thread j owning node j's frontier
// slot.  Because each depth's log-probs are sorted, a node's best remaining
// candidate is always its next rank, so the frontier holds one entry per node (B at
// most) and a node's slot simply moves to the next rank when it is popped.  Every
// slot's order is one 64-bit key, (order-preserving score << 32) | ~((parent << 16) |
// rank), 0 when empty, so a pop is a block-wide maximum: a warp reduction, one
// barrier (the warp maxima are double-buffered in shared memory, so no second barrier
// is needed), and every thread folding the 8 warp maxima itself.  After a pop only two
// threads act: the owner of the popped slot swaps in its next rank's key (computed
// ahead, off the critical path) and the new node's thread adds its first child, at
// once for w = 1 and when the round ends for w > 1.  The score comes back exactly
// from the winning key, so no other broadcast is needed.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kTreeMaxB = 256;
constexpr int kTreeThreads = 256;  // one frontier slot (node) per thread
constexpr int kTreeWarps = kTreeThreads / 32;

// Order-preserving image of a finite score (larger score -> larger value, never 0), and back.
__device__ __forceinline__ uint32_t score_key(float s)
{
    const uint32_t b = __float_as_uint(s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// A slot's order: larger score first, then smaller (parent, rank); 0 = empty.
__device__ __forceinline__ unsigned long long slot_order(float f, int parent, int rank)
{
    return ((unsigned long long)score_key(f) << 32) | (uint32_t)(~(((uint32_t)parent << 16) | (uint32_t)rank));
}

constexpr int kTreeSmemLp = 8192;  // log-prob tables up to this size are staged in shared memory

__global__ void __launch_bounds__(kTreeThreads) build_tree_kernel(const float *__restrict__ logp,
                                                                  const int32_t *__restrict__ tok, int Dmax, int K,
                                                                  int B, int w, int32_t *__restrict__ parent,
                                                                  int32_t *__restrict__ token,
                                                                  float *__restrict__ score, int32_t *status)
{
    __shared__ float sc[kTreeMaxB];
    __shared__ int16_t dep[kTreeMaxB], par[kTreeMaxB], rank[kTreeMaxB];
    __shared__ float s_lp[kTreeSmemLp];
    __shared__ unsigned long long s_best[2][kTreeWarps];
    __shared__ int s_bad;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float *g_lp = logp + (size_t)b * Dmax * K;
    const int32_t *tk = tok + (size_t)b * Dmax * K;

    pdl_wait_primary();
    pdl_launch_dependents();
    // each depth's log-probs finite and sorted best first; small tables go to shared memory
    const bool staged = Dmax * K <= kTreeSmemLp;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    bool bad = false;
    for (int t = tid; t < Dmax * K; t += kTreeThreads) {
        const float x = g_lp[t];
        if (!(fabsf(x) <= 3.0e38f)) bad = true;
        if (t % K + 1 < K && !(x >= g_lp[t + 1])) bad = true;
        if (staged) s_lp[t] = x;
    }
    if (bad) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        if (tid == 0) report_status(status, TV_ERR_INVALID_ARG);
        return;
    }
    const float *lp = staged ? s_lp : g_lp;

    // Thread j's slot is node j's next child.  key: its order now; nxt: the order of the
    // rank after it (ready before the pop that may take this one); my_f, my_d: node j's
    // score and depth; my_c: the rank the slot holds.
    unsigned long long key = 0ull, nxt = 0ull;
    float my_f = 0.f;
    int my_d = 0, my_c = 0;
    auto prepare_next = [&]() {  // the order of rank my_c + 1, or empty
        nxt = (my_c + 1 < K) ? slot_order(my_f + lp[(size_t)my_d * K + my_c + 1], tid, my_c + 1) : 0ull;
    };
    auto open_slot = [&]() {  // node tid (score my_f, depth my_d) offers its first child
        my_c = 0;
        if (my_d < Dmax) {
            key = slot_order(my_f + lp[(size_t)my_d * K], tid, 0);
            prepare_next();
        } else {
            key = 0ull;
        }
    };
    if (tid == 0) {
        sc[0] = 0.f;
        dep[0] = 0;
        par[0] = -1;
        rank[0] = 0;
        my_f = 0.f;
        my_d = 0;
        open_slot();
    }
    int made = 1, buf = 0;
    bool pending = false;  // this thread's node was made in the current round
    // A round takes up to w candidates (the popped slot moves to its next rank at once:
    // that sibling was a candidate when the round began), then the round's nodes offer
    // their first children; w = 1 is plain best-first expansion.
    while (made < B) {
        const int take = min(w, B - made);
        int got = 0;
        for (; got < take; ++got) {
            // block-wide maximum of the slot keys (warp maximum, then the 8 warp maxima)
            const uint32_t hi = (uint32_t)(key >> 32);
            const uint32_t whi = __reduce_max_sync(0xffffffffu, hi);
            const uint32_t wlo = __reduce_max_sync(0xffffffffu, hi == whi ? (uint32_t)key : 0u);
            if (lane == 0) s_best[buf][wid] = ((unsigned long long)whi << 32) | wlo;
            __syncthreads();
            unsigned long long top = s_best[buf][0];
#pragma unroll
            for (int k = 1; k < kTreeWarps; ++k) {
                const unsigned long long v = s_best[buf][k];
                top = v > top ? v : top;
            }
            buf ^= 1;
            if (top == 0ull) break;  // no candidate left this round
            const uint32_t t = ~(uint32_t)top;
            const int u = (int)(t >> 16), c = (int)(t & 0xFFFFu), i = made + got;
            const float f = key_score((uint32_t)(top >> 32));
            if (tid == u) {  // node i = (u, rank c); u's slot moves on to rank c + 1
                sc[i] = f;
                dep[i] = (int16_t)(my_d + 1);
                par[i] = (int16_t)u;
                rank[i] = (int16_t)c;
                key = nxt;
                my_c = c + 1;
                if (key != 0ull) prepare_next();
            }
            if (tid == i) {  // the new node: its children wait for the end of the round
                my_f = f;
                my_d = dep[u] + 1;
                pending = true;
            }
        }
        made += got;
        if (pending) {
            open_slot();
            pending = false;
        }
        if (got == 0) break;  // the round found no candidate at all: B exceeds the tree
    }
    __syncthreads();
    if (made < B && tid == 0) report_status(status, TV_ERR_INVALID_ARG);
    for (int i = tid; i < B; i += kTreeThreads) {
        const bool ok = i < made;
        parent[(size_t)b * B + i] = ok ? par[i] : -1;
        token[(size_t)b * B + i] = (ok && i > 0) ? tk[(size_t)(dep[i] - 1) * K + rank[i]] : -1;
        score[(size_t)b * B + i] = ok ? sc[i] : 0.f;
    }
}

cudaError_t launch_build_tree(const float *logp, const int32_t *tok, int nb, int Dmax, int K, int B, int w,
                              int32_t *parent, int32_t *token, float *score, int32_t *status, cudaStream_t stream)
{
    return launch_dependent(build_tree_kernel, dim3((unsigned)nb), dim3(kTreeThreads), 0, stream, logp, tok, Dmax, K,
                            B, w, parent, token, score, status);
}

}  // namespace tv
