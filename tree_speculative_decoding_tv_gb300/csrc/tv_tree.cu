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
// GPU form: one CTA of 256 threads per sequence, thread j owning node j's list of untaken
// children.  Because each depth's log-probs are sorted, that list is sorted best first, so
// the pool is a set of sorted lists.  The nodes are made in batches: a batch takes the
// pool's best candidates in one step, as many as the serial process would take before
// anything it creates could compete with them:
//   * within a w > 1 round nothing new enters the pool (the round's nodes offer their
//     children when it ends), so a batch is the round's best min(w, kTreeCap) candidates;
//   * for w = 1, a new node's candidates are all at most its first child, whose key
//     (score + the next depth's best log-prob, parent index at least `made`) bounds
//     everything a batch can create, and lies below x.  With T0 the largest bound of the
//     lists' heads and T1 the largest bound among the candidates above T0, the candidates
//     above T1 come out of the serial process before any created one (each is above every
//     bound of the candidates above it), so they form a batch.
// A batch larger than kTreeCap keeps its kTreeCap best (exact: rank counting, or a radix
// selection on the keys when there are more than kTreeCand candidates); each
// batch member's rank among the others gives its node index.  Keys order candidates
// exactly as the serial process does: (order-preserving score << 32) | ~((parent << 16) |
// rank).
#include <cuda_runtime.h>

#include <atomic>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kTreeMaxB = 256;
constexpr int kTreeThreads = kTreeMaxB;  // thread j: node j's list
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreeCap = 64;             // nodes made per batch at most
constexpr int kTreeCand = 128;           // candidates ranked directly (more go through a radix selection)
constexpr int kTreeKeys = 4;             // a list's next keys kept in registers
constexpr int kTreeSmemLp = 8192;        // log-prob tables up to this size are staged in shared memory

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

// A candidate's order: larger score first, then smaller (parent, rank); 0 = none.
__device__ __forceinline__ unsigned long long slot_order(float f, int parent, int rank)
{
    return ((unsigned long long)score_key(f) << 32) | (uint32_t)(~(((uint32_t)parent << 16) | (uint32_t)rank));
}

__device__ __forceinline__ unsigned long long warp_max64(unsigned long long v)
{
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0u);
    return ((unsigned long long)hi << 32) | lo;
}

struct TreeShared {
    float lp[kTreeSmemLp];
    float f[kTreeMaxB];                               // node score
    int d[kTreeMaxB], par[kTreeMaxB], rk[kTreeMaxB];  // depth, parent, rank
    int hn[kTreeMaxB];                                // next untaken child rank of each list
    unsigned long long buf[kTreeCap];                 // the batch (selection path)
    unsigned long long cand[kTreeCand];               // candidates above T, unordered
    unsigned long long heads[kTreeMaxB];              // w > 1: the lists' heads, unordered
    int red32[2][kTreeWarps];                         // block reductions (double-buffered)
    int ncand[2], nheads[2];  // counters of the gathers (double-buffered: see the loop)
    unsigned long long thr;
    uint32_t hist[256];
};

template <bool kStaged>
__global__ void __launch_bounds__(kTreeThreads) build_tree_kernel(const float *__restrict__ logp,
                                                                  const int32_t *__restrict__ tok, int Dmax, int K,
                                                                  int B, int w, int32_t *__restrict__ parent,
                                                                  int32_t *__restrict__ token,
                                                                  float *__restrict__ score, int32_t *status)
{
    extern __shared__ __align__(16) uint8_t tree_smem[];
    TreeShared &sh = *reinterpret_cast<TreeShared *>(tree_smem);
    const int b = blockIdx.x, j = threadIdx.x, lane = j & 31, wid = j >> 5;
    const float *g_lp = logp + (size_t)b * Dmax * K;
    const int32_t *tk = tok + (size_t)b * Dmax * K;
    auto LP = [&](int idx) -> float { return kStaged ? sh.lp[idx] : __ldg(g_lp + idx); };
    // Block reductions: one barrier each; the buffers alternate, so a buffer is written again
    // only after every thread has passed the barrier of the reduction in between.
    int rb = 0;
    auto block_max = [&](uint32_t v) {
        v = __reduce_max_sync(0xffffffffu, v);
        if (lane == 0) sh.red32[rb][wid] = (int)v;
        __syncthreads();
        uint32_t m0 = (uint32_t)sh.red32[rb][0], m1 = (uint32_t)sh.red32[rb][1];
#pragma unroll
        for (int k = 2; k < kTreeWarps; k += 2) {
            m0 = max(m0, (uint32_t)sh.red32[rb][k]);
            m1 = max(m1, (uint32_t)sh.red32[rb][k + 1]);
        }
        rb ^= 1;
        return max(m0, m1);
    };
    auto block_scan = [&](int v, int &total) {  // exclusive prefix over the threads, and the sum
        const int incl = warp_incl_scan(v, lane);
        if (lane == 31) sh.red32[rb][wid] = incl;
        __syncthreads();
        int before = 0;
        total = 0;
#pragma unroll
        for (int k = 0; k < kTreeWarps; ++k) {
            const int t = sh.red32[rb][k];
            before += k < wid ? t : 0;
            total += t;
        }
        rb ^= 1;
        return before + incl - v;
    };

    pdl_wait_primary();
    pdl_launch_dependents();
    // each depth's log-probs finite and sorted best first
    bool bad = false;
    for (int t = j; t < Dmax * K; t += kTreeThreads) {
        const float x = g_lp[t];
        if (!(fabsf(x) <= 3.0e38f)) bad = true;
        if (t % K + 1 < K && !(x >= g_lp[t + 1])) bad = true;
        if (kStaged) sh.lp[t] = x;
    }
    sh.hn[j] = K;
    if (j == 0) {
        sh.f[0] = 0.f;
        sh.d[0] = 0;
        sh.par[0] = -1;
        sh.rk[0] = 0;
        sh.hn[0] = 0;
        sh.ncand[0] = sh.ncand[1] = 0;
        sh.nheads[0] = sh.nheads[1] = 0;
    }
    if (__syncthreads_or(bad)) {
        if (j == 0) report_status(status, TV_ERR_INVALID_ARG);
        return;
    }

    // Node j's list: next rank hn, node score f, offset dk = depth * K of its children's
    // log-probs, its grandchildren's best log-prob c0 (NaN: none), and the keys of its next
    // kTreeKeys candidates kn (0: none; kn[0] is the head).
    const float kNone = __int_as_float(0x7fffffff);
    int hn = K, dk = 0;
    float f = 0.f, c0 = kNone;
    unsigned long long kn[kTreeKeys];
    auto key_at = [&](int c) { return slot_order(f + LP(dk + c), j, c); };
    auto load_keys = [&]() {
#pragma unroll
        for (int e = 0; e < kTreeKeys; ++e) kn[e] = hn + e < K ? key_at(hn + e) : 0ull;
    };
    if (j == 0) {
        hn = 0;
        c0 = Dmax > 1 ? LP(K) : kNone;
    }
    load_keys();
    // Calls fn(x) for the list's candidates x > lo, best first (at most kTreeCap: no more can
    // be taken from one list in a batch).
    auto each = [&](unsigned long long lo, auto &&fn) {
#pragma unroll
        for (int e = 0; e < kTreeKeys; ++e) {
            if (kn[e] <= lo) return;
            fn(kn[e]);
        }
        for (int c = hn + kTreeKeys, n = kTreeKeys; c < K && n < kTreeCap; ++c, ++n) {
            const unsigned long long x = key_at(c);
            if (x <= lo) return;
            fn(x);
        }
    };
    // The key bound on everything a new node made from candidate x of this list can offer:
    // its first child's score, with parent index `made`, the smallest a new node can have.
    // Only the high (score) word varies: bound_hi gives it, 1 standing for "no bound" (below
    // every score word), 0 for "no candidate".
    int made = 1;
    auto bound_hi = [&](unsigned long long x) -> uint32_t {
        if (x == 0ull) return 0u;
        return isnan(c0) ? 1u : score_key(key_score((uint32_t)(x >> 32)) + c0);
    };
    auto bound_key = [&](uint32_t hi) -> unsigned long long {  // hi > 1
        return ((unsigned long long)hi << 32) | (uint32_t)(~((uint32_t)made << 16));
    };
    // The q-th largest candidate above lo over all lists, by radix selection, 8 bits a pass
    // from the top, until the boundary bucket is taken whole: the keys >= the result are then
    // exactly q.  (Only for batches with more than kTreeCand candidates.)
    auto select = [&](unsigned long long lo, int q) {
        unsigned long long prefix = 0ull;
        int need = q;
        for (int shift = 56; shift >= 0; shift -= 8) {
            const unsigned long long hmask = shift == 56 ? 0ull : (~0ull << (shift + 8));
            sh.hist[j] = 0u;
            __syncthreads();
            each(lo, [&](unsigned long long x) {
                if ((x & hmask) == prefix) atomicAdd(&sh.hist[(uint32_t)(x >> shift) & 255u], 1u);
            });
            __syncthreads();
            // every warp finds the bucket from the whole histogram
            uint32_t h[8], sum = 0;  // lane l holds bins 255 - 8l - k: highest bins first
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                h[k] = sh.hist[255 - 8 * lane - k];
                sum += h[k];
            }
            const int incl = warp_incl_scan((int)sum, lane);
            const int excl = incl - (int)sum;
            const int src = __ffs(__ballot_sync(0xffffffffu, excl < need && need <= incl)) - 1;
            int bin = 0, above = 0, inbin = 0;
            if (lane == src) {
                int acc = excl;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (inbin == 0 && acc + (int)h[k] >= need) {
                        bin = 255 - 8 * lane - k;
                        above = acc;
                        inbin = (int)h[k];
                    }
                    acc += (int)h[k];
                }
            }
            bin = __shfl_sync(0xffffffffu, bin, src);
            above = __shfl_sync(0xffffffffu, above, src);
            inbin = __shfl_sync(0xffffffffu, inbin, src);
            need -= above;
            prefix |= (unsigned long long)bin << shift;
            __syncthreads();  // the histogram is read before the next pass clears it
            if (inbin == need) break;
        }
        return prefix;
    };

    const bool one = w == 1;
    int quota = 0, round0 = 1;  // w > 1: nodes still to take in this round, its first node
    // Every pass makes at least one node or ends a round, so 2 B passes always suffice; the
    // cap only guards against a broken invariant (reported, never a hang).
    for (int pass = 0; made < B; ++pass) {
        if (pass > 2 * kTreeMaxB + 2) {
            if (j == 0) report_status(status, TV_ERR_INVALID_ARG);
            break;
        }
        // this pass's gather counters; the other pair (last read before the previous pass's
        // final barrier) is cleared for the next pass, which gathers only after a barrier
        const int cb = pass & 1;
        if (j == 0) {
            sh.ncand[cb ^ 1] = 0;
            sh.nheads[cb ^ 1] = 0;
        }
        if (!one && quota == 0) {  // a round begins: the previous round's nodes offer their children
            if (j >= round0 && j < made && dk < Dmax * K) {
                hn = 0;
                load_keys();
                sh.hn[j] = 0;
            }
            quota = min(w, B - made);
            round0 = made;
        }
        const int want = one ? B - made : quota;

        // T: the batch is the q best candidates above T
        unsigned long long T = 0ull;
        bool empty;
        if (one) {
            // A bound is below its candidate, so no head outside the largest batch has a bound
            // above that batch's largest bound, and T0, the largest bound of the heads, is at
            // most it: the candidates above T0 include that batch.  The largest bound among
            // them, T, is then at least its largest bound, and the candidates above T form a
            // batch (each is above every bound of the candidates above it).
            const uint32_t a = block_max(bound_hi(kn[0]));
            empty = a == 0u;
            const unsigned long long t0 = a > 1u ? bound_key(a) : 0ull;
            uint32_t m = 1u;
            each(t0, [&](unsigned long long x) { m = max(m, bound_hi(x)); });
            m = block_max(m);
            T = m > 1u ? bound_key(m) : 0ull;
        } else {
            // the round's best min(want, kTreeCap) candidates lie at or above its qh-th best head
            if (kn[0] != 0ull) sh.heads[atomicAdd(&sh.nheads[cb], 1)] = kn[0];
            __syncthreads();
            const int nh = sh.nheads[cb];
            empty = nh == 0;
            const int qh = min(min(want, kTreeCap), nh);
            if (nh > qh) {
                if (kn[0] != 0ull) {
                    // eight independent counts, so the shared-memory loads overlap
                    const unsigned long long v = kn[0];
                    int r0 = 0, r1 = 0, r2 = 0, r3 = 0, r4 = 0, r5 = 0, r6 = 0, r7 = 0;
                    int e = 0;
                    for (; e + 8 <= nh; e += 8) {
                        r0 += sh.heads[e] > v;
                        r1 += sh.heads[e + 1] > v;
                        r2 += sh.heads[e + 2] > v;
                        r3 += sh.heads[e + 3] > v;
                        r4 += sh.heads[e + 4] > v;
                        r5 += sh.heads[e + 5] > v;
                        r6 += sh.heads[e + 6] > v;
                        r7 += sh.heads[e + 7] > v;
                    }
                    for (; e < nh; ++e) r0 += sh.heads[e] > v;
                    const int r = ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
                    if (r == qh - 1) sh.thr = v - 1ull;
                }
                __syncthreads();
                T = sh.thr;
            }
        }
        if (empty) {
            if (!one && made > round0) {  // the pool ran dry: the round ends early
                quota = 0;
                continue;
            }
            break;  // nothing left at all: B exceeds the tree
        }

        // gather the candidates above T (unordered); a member's rank among them is its place
        int cnt = 0;
        each(T, [&](unsigned long long x) {
            const int idx = atomicAdd(&sh.ncand[cb], 1);
            if (idx < kTreeCand) sh.cand[idx] = x;
            ++cnt;
        });
        __syncthreads();
        const int total = sh.ncand[cb];
        const int q = min(min(total, want), kTreeCap);
        if (q <= 0) {  // cannot happen (the best candidate is always above T); never loop on it
            if (j == 0) report_status(status, TV_ERR_INVALID_ARG);
            break;
        }
        if (total <= kTreeCand) {
            if (j < total) {
                const unsigned long long v = sh.cand[j];
                int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
                int e = 0;
                for (; e + 4 <= total; e += 4) {
                    r0 += sh.cand[e] > v;
                    r1 += sh.cand[e + 1] > v;
                    r2 += sh.cand[e + 2] > v;
                    r3 += sh.cand[e + 3] > v;
                }
                for (; e < total; ++e) r0 += sh.cand[e] > v;
                const int r = (r0 + r1) + (r2 + r3);
                if (r < q) {
                    const uint32_t tl = ~(uint32_t)v;
                    const int u = (int)(tl >> 16), c = (int)(tl & 0xFFFFu), i = made + r;
                    const int d = sh.d[u] + 1;
                    sh.f[i] = key_score((uint32_t)(v >> 32));
                    sh.d[i] = d;
                    sh.par[i] = u;
                    sh.rk[i] = c;
                    sh.hn[i] = (one && d < Dmax) ? 0 : K;
                    atomicMax(&sh.hn[u], c + 1);  // a list's taken candidates are a prefix of it
                }
            }
        } else {
            // too many to rank directly: select the q-th largest, gather the q, rank them
            const unsigned long long kappa = select(T, q);
            cnt = 0;
            each(kappa - 1ull, [&](unsigned long long) { ++cnt; });
            int tot = 0;
            int off = block_scan(cnt, tot);
            each(kappa - 1ull, [&](unsigned long long x) { sh.buf[off++] = x; });
            __syncthreads();
            if (j < q) {
                const unsigned long long v = sh.buf[j];
                int r = 0;
                for (int e = 0; e < q; ++e) r += sh.buf[e] > v;
                const uint32_t tl = ~(uint32_t)v;
                const int u = (int)(tl >> 16), c = (int)(tl & 0xFFFFu), i = made + r;
                const int d = sh.d[u] + 1;
                sh.f[i] = key_score((uint32_t)(v >> 32));
                sh.d[i] = d;
                sh.par[i] = u;
                sh.rk[i] = c;
                sh.hn[i] = (one && d < Dmax) ? 0 : K;
                atomicMax(&sh.hn[u], c + 1);
            }
        }
        __syncthreads();
        if (j < made) {  // a list that advanced moves on to its next candidates
            const int nh = sh.hn[j];
            if (nh != hn) {
                hn = nh;
                load_keys();
            }
        } else if (j < made + q) {  // this thread's node was just made
            f = sh.f[j];
            const int d = sh.d[j];
            dk = d * K;
            c0 = d + 1 < Dmax ? LP(dk + K) : kNone;
            hn = sh.hn[j];
            load_keys();
        }
        made += q;
        if (!one) quota -= q;
    }
    __syncthreads();
    if (made < B && j == 0) report_status(status, TV_ERR_INVALID_ARG);
    for (int i = j; i < B; i += kTreeThreads) {
        const bool ok = i < made;
        parent[(size_t)b * B + i] = ok ? sh.par[i] : -1;
        token[(size_t)b * B + i] = (ok && i > 0) ? tk[(size_t)(sh.d[i] - 1) * K + sh.rk[i]] : -1;
        score[(size_t)b * B + i] = ok ? sh.f[i] : 0.f;
    }
}

cudaError_t launch_build_tree(const float *logp, const int32_t *tok, int nb, int Dmax, int K, int B, int w,
                              int32_t *parent, int32_t *token, float *score, int32_t *status, cudaStream_t stream)
{
    const bool staged = (long long)Dmax * K <= kTreeSmemLp;
    auto kernel = staged ? build_tree_kernel<true> : build_tree_kernel<false>;
    static std::atomic<uint64_t> opted_in[2];  // the shared-memory opt-in, once per device and kernel
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (!bit || !(opted_in[staged].load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(TreeShared));
        if (e != cudaSuccess) return e;
        if (bit) opted_in[staged].fetch_or(bit, std::memory_order_relaxed);
    }
    return launch_dependent(kernel, dim3((unsigned)nb), dim3(kTreeThreads), sizeof(TreeShared), stream, logp, tok, Dmax, K, B,
                            w, parent, token, score, status);
}

}  // namespace tv
