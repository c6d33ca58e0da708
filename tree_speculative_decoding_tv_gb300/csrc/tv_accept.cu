// Vocab argmax and greedy acceptance walk.
//
// The pages speak of accepted tokens and longer accepted prefixes (JETFLOW
// summary, §3 item 2 and §4) without stating a rule; the rule implemented is
// the greedy one: node i >= 1 is accepted iff its parent is accepted and its
// draft token equals the target argmax at the parent; the deepest accepted
// node wins, ties to the smallest index.
//
// argmax (kernel 1): the logits are cut into (row, 4096-element chunk) units, one
// warp per unit.  A lane holds 16 16-byte vectors of its unit in registers (all in
// flight at once); bf16x2 NaN-propagating max instructions reduce them (about one per
// two logits), the warp agrees on the unit's maximum with shuffles, and only the lanes
// holding it look for its first position.  Each unit folds into a 64-bit
// order-preserving key (value rank, then the smaller index).  The units of all rows,
// row-major, are cut into equal contiguous shares, one per warp of a grid of two CTAs
// per SM, so every warp streams the same number of 8 KB units however many rows there
// are; a warp combines its units of one row in registers and adds the result to the
// row's key in the workspace with one 64-bit atomicMax per row it touches.  The keys
// start at zero, below every real key, and the acceptance kernel sets each back to
// zero once it has read it, so no memset runs between calls.
//
// accept (kernel 2): one CTA per sequence, one thread per node, launched as a
// programmatic dependent of the argmax.  The tree inputs (parent, draft, the
// mask rows) are loaded into shared memory while the argmax still runs; after
// the dependency wait each thread reads its row's key, ok[] is packed into W
// ballot words, node i is accepted iff (mask[i] & ~ok) == 0 (the root counts as
// ok), the best (depth, -index) key is a block max, and the path is read off
// the chosen node's mask bits in ascending order.
//
// fused (tv_accept_fused, one kernel): CTAs that own whole rows (R = max(1, 8 / chunks
// per row) at a time, whose units their 8 warps share, combined in shared memory into
// one key per row stored with a plain store), and after a CTA
// stores a row group's keys it adds the group's row count to a per-sequence
// counter in the workspace; the CTA whose addition completes sequence b's B rows
// resets the counter and runs b's acceptance walk itself (a fence orders every
// CTA's keys before its addition, and the walking CTA's fence after it before
// it reads them).  Nothing waits on another CTA.  Without a mask the walking CTA
// builds node i's ancestor bits in shared memory by walking i's root path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "tv_argmax.cuh"
#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kArgThreads = 256;
constexpr int kArgVec = 16;                   // 16-byte vectors per lane per unit
constexpr int kArgChunk = 32 * kArgVec * 8;   // logits per unit (8 KB): one warp
constexpr int kArgCtasPerSm = 2;  // resident CTAs per SM at the kernel's register use
constexpr int kMaxB = 256;
constexpr int kMaxW = kMaxB / 32;

// Shared memory of one acceptance walk (one sequence, one thread per node).
struct AcceptSmem {
    int am[kMaxB];
    int16_t par[kMaxB];  // the fused walk's parent array (mask built in-kernel)
    uint32_t mask[kMaxB * kMaxW];
    uint32_t ok[kMaxW];
    int best[kMaxB / 32];
    int bad;
};

// The walk proper, once s.am (every row's argmax) and s.mask (every node's ancestor
// bits) are in shared memory and visible: p and d are this thread's parent and draft
// token (thread i = node i).
__device__ __forceinline__ void accept_core(AcceptSmem &s, int b, int B, int W, int p, int d,
                                            int32_t *__restrict__ n_acc, int32_t *__restrict__ path,
                                            int32_t *__restrict__ bonus, int32_t *status)
{
    const int i = threadIdx.x;
    const int lane = i & 31, wid = i >> 5;
    bool ok = true;
    if (i > 0 && i < B) {
        if (p < 0 || p >= i) {
            ok = false;
            s.bad = 1;
        } else {
            ok = d == s.am[p];
        }
    }
    const uint32_t okw = __ballot_sync(0xffffffffu, ok);
    if (lane == 0 && wid < kMaxW) s.ok[wid] = okw;
    __syncthreads();

    int key = -1;  // depth * 512 + (511 - node) of an accepted node
    if (i < B) {
        bool acc = true;
        int bits = 0;
        for (int w = 0; w < W; ++w) {
            const uint32_t mw = s.mask[i * W + w];
            acc = acc && ((mw & ~s.ok[w]) == 0u);
            bits += __popc(mw);
        }
        if (acc) key = (bits - 1) * 512 + (511 - i);
    }
    key = __reduce_max_sync(0xffffffffu, key);
    if (lane == 0) s.best[wid] = key;
    __syncthreads();
    int top = s.best[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) top = max(top, s.best[w]);
    const int vstar = top >= 0 ? 511 - (top & 511) : 0;
    const int dep = top >= 0 ? (top >> 9) : 0;
    const uint32_t *vmask = s.mask + vstar * W;

    if (i < B) {
        const int w = i >> 5;
        const uint32_t mw = vmask[w];
        if ((mw >> lane) & 1u) {
            int before = __popc(mw & ((1u << lane) - 1u));
            for (int k = 0; k < w; ++k) before += __popc(vmask[k]);
            path[(size_t)b * B + before] = i;
        }
        if (i > dep) path[(size_t)b * B + i] = -1;
    }
    if (i == 0) {
        n_acc[b] = dep;
        bonus[b] = s.am[vstar];
        if (s.bad) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
    }
}

// Outputs for a sequence whose parent array is not topological (no mask to walk):
// the root alone is accepted; s.am must hold the rows' argmax.
__device__ __forceinline__ void accept_bad_tree(const AcceptSmem &s, int b, int B, int32_t *__restrict__ n_acc,
                                                int32_t *__restrict__ path, int32_t *__restrict__ bonus,
                                                int32_t *status)
{
    const int i = threadIdx.x;
    if (i < B) path[(size_t)b * B + i] = (i == 0) ? 0 : -1;
    if (i == 0) {
        n_acc[b] = 0;
        bonus[b] = s.am[0];
        report_status(status, TV_ERR_NOT_TOPOLOGICAL);
    }
}

// Node i's ancestor bits from a walk up its root path in shared memory (s.par must be
// staged and topological): the mask build folded into the acceptance.
__device__ __forceinline__ void accept_rows_from_parents(AcceptSmem &s, int B, int W)
{
    const int i = threadIdx.x;
    if (i < B) {
        uint32_t *row = s.mask + i * W;
        for (int w = 0; w < W; ++w) row[w] = 0u;
        for (int j = i; j >= 0; j = s.par[j]) row[j >> 5] |= 1u << (j & 31);
    }
}

// Sequence b's acceptance inside the fused kernel, run by the CTA that completed b's
// keys (every CTA's keys are visible to it: see the fences in the caller).  With no
// mask, node i's ancestor bits come from a walk up its root path, after the parent
// array has been checked (a bad one reports TV_ERR_NOT_TOPOLOGICAL and gives the
// root alone as the accepted path).
__device__ void fused_walk(AcceptSmem &s, int b, int B, int W, const unsigned long long *__restrict__ best,
                           const int32_t *__restrict__ draft, const int32_t *__restrict__ parent,
                           const uint32_t *__restrict__ mask, int32_t *__restrict__ am,
                           int32_t *__restrict__ n_acc, int32_t *__restrict__ path, int32_t *__restrict__ bonus,
                           int32_t *status)
{
    const int i = threadIdx.x;
    int p = -1, d = 0;
    bool bad = false;
    if (i < B) {
        p = parent[(size_t)b * B + i];
        d = draft[(size_t)b * B + i];
        bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
        const unsigned long long top = __ldcg(best + (size_t)b * B + i);
        const int a = (int)(0xFFFFFFFFu - (uint32_t)top);
        s.am[i] = a;
        am[(size_t)b * B + i] = a;
    }
    if (i == 0) s.bad = 0;
    if (mask) {
        if (i < B)
            for (int w = 0; w < W; ++w) s.mask[i * W + w] = mask[((size_t)b * B + i) * W + w];
    } else {
        if (i < B) s.par[i] = (int16_t)p;
        if (__syncthreads_or(bad)) {
            accept_bad_tree(s, b, B, n_acc, path, bonus, status);
            return;
        }
        accept_rows_from_parents(s, B, W);
    }
    __syncthreads();
    accept_core(s, b, B, W, p, d, n_acc, path, bonus, status);
}

// One unit: logits [lo, min(lo + kArgChunk, V)) of one row, reduced by one warp to the
// 64-bit order-preserving key of its maximum (value rank, then the smaller index); the
// result is the same in every lane.  Each lane holds kArgVec 16-byte vectors in
// registers (all loads in flight at once) and folds them as a tree of bf16x2 maxima,
// keeping each vector's maximum; the warp agrees on the unit's maximum with one integer
// max-reduction of its rank, the lanes holding it find their first position in two
// steps (first vector whose maximum matches, then the element inside it), and one
// integer min-reduction picks the smallest.  32-bit index arithmetic.
__device__ __forceinline__ unsigned long long unit_key(const uint16_t *__restrict__ row, int lo, int V, int lane)
{
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int hi = min(lo + kArgChunk, V);

    // scalar head up to the first 16-byte boundary, 16-byte vectors, scalar tail
    const int head = min((int)(((16u - ((uint32_t)(uintptr_t)(row + lo) & 15u)) & 15u) >> 1), hi - lo);
    const int vstart = lo + head;
    const int nvec = (hi - vstart) >> 3;
    const int tail = vstart + nvec * 8;
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + vstart);
    uint4 v[kArgVec];
    if (nvec > 0) {
#pragma unroll
        for (int k = 0; k < kArgVec; ++k) v[k] = ld_stream_v4(vp + min(lane + k * 32, nvec - 1));
        // dependency points: every load is issued before any of them is used
        asm volatile("" : "+r"(v[0].x), "+r"(v[0].y), "+r"(v[0].z), "+r"(v[0].w), "+r"(v[1].x), "+r"(v[1].y),
                     "+r"(v[1].z), "+r"(v[1].w), "+r"(v[2].x), "+r"(v[2].y), "+r"(v[2].z), "+r"(v[2].w),
                     "+r"(v[3].x), "+r"(v[3].y), "+r"(v[3].z), "+r"(v[3].w), "+r"(v[4].x), "+r"(v[4].y),
                     "+r"(v[4].z), "+r"(v[4].w), "+r"(v[5].x), "+r"(v[5].y), "+r"(v[5].z), "+r"(v[5].w),
                     "+r"(v[6].x), "+r"(v[6].y), "+r"(v[6].z), "+r"(v[6].w), "+r"(v[7].x), "+r"(v[7].y),
                     "+r"(v[7].z), "+r"(v[7].w));
        asm volatile("" : "+r"(v[8].x), "+r"(v[8].y), "+r"(v[8].z), "+r"(v[8].w), "+r"(v[9].x), "+r"(v[9].y),
                     "+r"(v[9].z), "+r"(v[9].w), "+r"(v[10].x), "+r"(v[10].y), "+r"(v[10].z), "+r"(v[10].w),
                     "+r"(v[11].x), "+r"(v[11].y), "+r"(v[11].z), "+r"(v[11].w), "+r"(v[12].x), "+r"(v[12].y),
                     "+r"(v[12].z), "+r"(v[12].w), "+r"(v[13].x), "+r"(v[13].y), "+r"(v[13].z), "+r"(v[13].w),
                     "+r"(v[14].x), "+r"(v[14].y), "+r"(v[14].z), "+r"(v[14].w), "+r"(v[15].x), "+r"(v[15].y),
                     "+r"(v[15].z), "+r"(v[15].w));
    }
    const bool has_head = lane < head, has_tail = lane < hi - tail;
    const float xh = has_head ? bf16_bits_to_float(row[lo + lane]) : NEG_INF;
    const float xt = has_tail ? bf16_bits_to_float(row[tail + lane]) : NEG_INF;

    // lane maximum: a bf16x2 tree over the vectors (clamped duplicates of the last
    // vector do not change it); the vector maxima stay for the search
    __nv_bfloat162 vm[kArgVec];
#pragma unroll
    for (int k = 0; k < kArgVec; ++k) vm[k] = vec_max2(v[k]);
    __nv_bfloat162 t[kArgVec / 2];
#pragma unroll
    for (int k = 0; k < kArgVec / 2; ++k) t[k] = __hmax2_nan(vm[2 * k], vm[2 * k + 1]);
#pragma unroll
    for (int w = kArgVec / 4; w > 0; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) t[k] = __hmax2_nan(t[2 * k], t[2 * k + 1]);
    const float vmax = nvec > 0 ? __bfloat162float(__hmax_nan(t[0].x, t[0].y)) : NEG_INF;
    const float tm = max_nan(max_nan(vmax, xh), xt);
    const uint32_t r = value_rank(tm);
    const uint32_t wr = __reduce_max_sync(0xffffffffu, r);

    // first position of the unit maximum in this lane (index order: head, vectors, tail)
    uint32_t idx = 0x7fffffffu;
    if (r == wr) {
        const bool nan = tm != tm;
        if (has_head && (nan ? (xh != xh) : (xh == tm))) {
            idx = lo + lane;
        } else {
            int kf = -1;
#pragma unroll
            for (int k = kArgVec - 1; k >= 0; --k) {
                const float x = __bfloat162float(__hmax_nan(vm[k].x, vm[k].y));
                if (lane + k * 32 < nvec && (nan ? (x != x) : (x == tm))) kf = k;
            }
            if (kf >= 0) {
                uint4 w = v[0];
#pragma unroll
                for (int k = 1; k < kArgVec; ++k)
                    if (k == kf) w = v[k];
                const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
                int e_first = 7;
#pragma unroll
                for (int e = 7; e >= 0; --e) {
                    const float x = bf16_bits_to_float((w4[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
                    if (nan ? (x != x) : (x == tm)) e_first = e;
                }
                idx = vstart + (lane + kf * 32) * 8 + e_first;
            } else if (has_tail) {
                idx = tail + lane;
            }
        }
    }
    idx = __reduce_min_sync(0xffffffffu, idx);
    return ((unsigned long long)wr << 32) | (0xFFFFFFFFu - idx);
}

// One unit = kArgChunk logits of one row = one warp: each lane holds kArgVec
// 16-byte vectors in registers (all loads in flight at once) and folds them as
// a tree of bf16x2 maxima, keeping each vector's maximum; the warp agrees on the
// unit's maximum with one integer max-reduction of its rank, the lanes holding
// it find their first position in two steps (first vector whose maximum
// matches, then the element inside it), and one integer min-reduction picks the
// smallest.  No block-level synchronisation; 32-bit index arithmetic.
// What the fused kernel needs for the acceptance walks (unused by the plain argmax).
struct FusedAccept {
    unsigned int *counters;  // [nb] rows whose keys are stored so far; zero between calls
    int B, W;
    const int32_t *draft, *parent;
    const uint32_t *mask;  // may be null
    int32_t *am, *n_acc, *path, *bonus, *status;
};

template <bool kFused>
__global__ void __launch_bounds__(kArgThreads) argmax_rows_kernel(const uint16_t *__restrict__ logits, int V,
                                                                  int nchunk, int R, int rows,
                                                                  unsigned long long *__restrict__ best,
                                                                  FusedAccept fa)
{
    __shared__ unsigned long long s_key[kArgThreads / 32];  // R <= 8 rows per group
    static_assert(kArgChunk == 32 * kArgVec * 8, "one warp per unit");
    static_assert(kArgVec == 16, "the dependency points below list 16 vectors");
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    pdl_wait_primary();  // the logits may come from the previous kernel in the stream
    pdl_launch_dependents();
    if constexpr (kFused) {
        // whichever CTA walks a sequence reads its tree inputs: start them towards L2 now
        const int b0 = blockIdx.x * R / fa.B;
        const int b1 = min(rows - 1, blockIdx.x * R + R - 1) / fa.B;
        for (int bb = b0; bb <= b1; ++bb) {
            const int lines_pd = (fa.B * 4 + 127) / 128, lines_m = fa.mask ? (fa.B * fa.W * 4 + 127) / 128 : 0;
            for (int t = threadIdx.x; t < 2 * lines_pd + lines_m; t += kArgThreads) {
                const char *a = t < lines_pd ? reinterpret_cast<const char *>(fa.parent + (size_t)bb * fa.B) + 128 * t
                              : t < 2 * lines_pd
                                  ? reinterpret_cast<const char *>(fa.draft + (size_t)bb * fa.B) + 128 * (t - lines_pd)
                                  : reinterpret_cast<const char *>(fa.mask + (size_t)bb * fa.B * fa.W) +
                                        128 * (t - 2 * lines_pd);
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
            }
        }
    }

    for (int r0 = blockIdx.x * R; r0 < rows; r0 += gridDim.x * R) {
      const int nr = min(R, rows - r0);
      if (threadIdx.x < kArgThreads / 32) s_key[threadIdx.x] = 0ull;  // below every real key
      __syncthreads();
      for (int u = wid; u < nr * nchunk; u += kArgThreads / 32) {
        const int lr = u / nchunk;
        const int row_id = r0 + lr;
        const int lo = (u - lr * nchunk) * kArgChunk;
        const unsigned long long key = unit_key(logits + (size_t)row_id * V, lo, V, lane);
        if (lane == 0) atomicMax(&s_key[lr], key);
      }
      __syncthreads();
      if (threadIdx.x < nr) best[r0 + threadIdx.x] = s_key[threadIdx.x];
      if constexpr (kFused) {
          __shared__ AcceptSmem s_acc;
          __shared__ int s_walk[kArgThreads / 32], s_nwalk;
          if ((int)threadIdx.x < nr) __threadfence();  // this CTA's keys before its counter additions
          if (threadIdx.x == 0) s_nwalk = 0;
          __syncthreads();
          // the sequences this group's rows belong to (at most nr <= 8)
          const int b0 = r0 / fa.B, bb = b0 + (int)threadIdx.x;
          if (bb <= (r0 + nr - 1) / fa.B) {
              const unsigned c = (unsigned)(min(r0 + nr, (bb + 1) * fa.B) - max(r0, bb * fa.B));
              if (atomicAdd(&fa.counters[bb], c) + c == (unsigned)fa.B) {  // b's last rows: walk it
                  fa.counters[bb] = 0u;
                  s_walk[atomicAdd(&s_nwalk, 1)] = bb;
              }
          }
          __syncthreads();
          const int nw = s_nwalk;
          if (nw > 0) __threadfence();  // every other CTA's keys of those sequences from here
          for (int k = 0; k < nw; ++k) {
              fused_walk(s_acc, s_walk[k], fa.B, fa.W, best, fa.draft, fa.parent, fa.mask, fa.am, fa.n_acc,
                         fa.path, fa.bonus, fa.status);
              __syncthreads();
          }
      }
      __syncthreads();  // s_key is reset for the next group only after it was read
    }
}

// tv_accept's argmax: the (row, chunk) units of all rows, row-major, are cut into equal
// contiguous shares, one per warp of the grid, so every warp streams the same number
// of 8 KB units whatever the row count (no tail of SMs holding an extra row).  A warp
// folds the units of one row into a register key and adds it to the row's key with one
// 64-bit atomicMax when it moves to the next row or ends; the keys start at zero (below
// every real key) and the acceptance kernel sets them back to zero after reading them.
__global__ void __launch_bounds__(kArgThreads) argmax_span_kernel(const uint16_t *__restrict__ logits, int V,
                                                                  int nchunk, long long units,
                                                                  unsigned long long *__restrict__ keys)
{
    const int lane = threadIdx.x & 31;
    const long long W = (long long)gridDim.x * (kArgThreads / 32);
    const long long w = (long long)blockIdx.x * (kArgThreads / 32) + (threadIdx.x >> 5);
    pdl_wait_primary();  // the logits may come from the previous kernel in the stream
    pdl_launch_dependents();
    const long long u0 = units * w / W, u1 = units * (w + 1) / W;
    int row = -1;
    unsigned long long best = 0ull;
    for (long long u = u0; u < u1; ++u) {
        const int r = (int)(u / nchunk);
        const int c = (int)(u - (long long)r * nchunk);
        if (r != row) {
            if (row >= 0 && lane == 0) atomicMax(keys + row, best);
            row = r;
            best = 0ull;
        }
        const unsigned long long k = unit_key(logits + (size_t)r * V, c * kArgChunk, V, lane);
        best = k > best ? k : best;
    }
    if (row >= 0 && lane == 0) atomicMax(keys + row, best);
}

__global__ void __launch_bounds__(kMaxB) accept_kernel(unsigned long long *__restrict__ best,
                                                       const int32_t *__restrict__ draft,
                                                       const int32_t *__restrict__ parent,
                                                       const uint32_t *__restrict__ mask, int B, int W,
                                                       int32_t *__restrict__ am, int32_t *__restrict__ n_acc,
                                                       int32_t *__restrict__ path, int32_t *__restrict__ bonus,
                                                       int32_t *status)
{
    __shared__ AcceptSmem s;
    const int b = blockIdx.x;
    const int i = threadIdx.x;

    // The argmax CTAs let this kernel launch only after their own dependency wait, so
    // everything before the argmax (the tree inputs) is complete and is read while the
    // argmax still runs; only the keys wait for it.
    int p = -1, d = 0;
    bool bad = false;
    if (i < B) {
        p = parent[(size_t)b * B + i];
        d = draft[(size_t)b * B + i];
        if (mask) {
            uint32_t mrow[kMaxW];
#pragma unroll
            for (int w = 0; w < kMaxW; ++w)  // all row words in flight at once
                if (w < W) mrow[w] = mask[((size_t)b * B + i) * W + w];
#pragma unroll
            for (int w = 0; w < kMaxW; ++w)
                if (w < W) s.mask[i * W + w] = mrow[w];
        } else {
            bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
            s.par[i] = (int16_t)p;
        }
    }
    if (i == 0) s.bad = 0;
    // without a mask array the rows are built here, while the argmax still runs
    const bool bad_tree = !mask && __syncthreads_or(bad);
    if (!mask && !bad_tree) accept_rows_from_parents(s, B, W);
    pdl_wait_primary();  // the argmax keys are complete from here on

    // every row's argmax is the low half of its key: 0xFFFFFFFF - index; the key goes back
    // to zero for the next call (the argmax combines into zeroed keys)
    if (i < B) {
        const unsigned long long top = __ldcg(best + (size_t)b * B + i);
        best[(size_t)b * B + i] = 0ull;
        const int a = (int)(0xFFFFFFFFu - (uint32_t)top);
        s.am[i] = a;
        am[(size_t)b * B + i] = a;
    }
    __syncthreads();
    if (bad_tree) {
        accept_bad_tree(s, b, B, n_acc, path, bonus, status);
        return;
    }
    accept_core(s, b, B, W, p, d, n_acc, path, bonus, status);
}

size_t accept_workspace_bytes(int V, int B, int nb)
{
    (void)V;
    return (size_t)nb * B * sizeof(unsigned long long);
}

cudaError_t launch_accept(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                          const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                          int32_t *bonus, int32_t *status, void *workspace, int num_sms, cudaStream_t stream)
{
    const int nchunk = (V + kArgChunk - 1) / kArgChunk;
    const long long units = (long long)nb * B * nchunk;
    long long grid = (long long)num_sms * kArgCtasPerSm;
    const long long need = (units + kArgThreads / 32 - 1) / (kArgThreads / 32);  // at least one unit per warp
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    unsigned long long *best = static_cast<unsigned long long *>(workspace);
    cudaError_t e = launch_dependent(argmax_span_kernel, dim3((unsigned)grid), dim3(kArgThreads), 0, stream, logits, V,
                                     nchunk, units, best);
    if (e != cudaSuccess) return e;
    const int W = (B + 31) / 32;
    // its launch overlaps the argmax tail; it waits before reading the keys
    return launch_dependent(accept_kernel, dim3((unsigned)nb), dim3(kMaxB), 0, stream, best, draft, parent, mask, B, W,
                            am, n_acc, path, bonus, status);
}

size_t accept_fused_workspace_bytes(int V, int B, int nb)
{
    return accept_workspace_bytes(V, B, nb) + (size_t)nb * sizeof(unsigned int);
}

cudaError_t launch_accept_fused(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                                const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                                int32_t *bonus, int32_t *status, void *workspace, int num_sms, cudaStream_t stream)
{
    const int nchunk = (V + kArgChunk - 1) / kArgChunk;
    const int rows = nb * B;
    const int wpc = kArgThreads / 32;
    const int R = nchunk >= wpc ? 1 : wpc / nchunk;
    long long grid = (long long)num_sms * kArgCtasPerSm;
    const long long need = ((long long)rows + R - 1) / R;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    unsigned long long *best = static_cast<unsigned long long *>(workspace);
    FusedAccept fa;
    fa.counters = reinterpret_cast<unsigned int *>(best + (size_t)rows);
    fa.B = B;
    fa.W = (B + 31) / 32;
    fa.draft = draft;
    fa.parent = parent;
    fa.mask = mask;
    fa.am = am;
    fa.n_acc = n_acc;
    fa.path = path;
    fa.bonus = bonus;
    fa.status = status;
    return launch_dependent(argmax_rows_kernel<true>, dim3((unsigned)grid), dim3(kArgThreads), 0, stream, logits, V,
                            nchunk, R, rows, best, fa);
}

// ------------------------------------------------------ allocation-free variant

// Scratch of tv_accept_noalloc: one 8-byte argmax key per logits row, for at most
// TV_ACCEPT_NOALLOC_MAX_ROWS rows (64 KB).  It lives in the library image, so every
// GPU that loads the library holds it until the process exits, and every call of
// tv_accept_noalloc on that GPU shares it.
static __device__ __align__(256) unsigned long long g_noalloc_keys[TV_ACCEPT_NOALLOC_MAX_ROWS];

// The device address of g_noalloc_keys in the current context.  Host code only sees a
// host-side stand-in under that name, so the address is looked up with
// cudaGetSymbolAddress (with the device current) the first time a context calls, and
// cached per device together with the context's unique id: a context created after
// cudaDeviceReset loads the module again, possibly elsewhere, and gets a fresh lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

static unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(a);
            get_id = reinterpret_cast<CtxGetIdFn>(b);
        }
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;  // unknown: the lookup is then repeated on every call
}

static cudaError_t noalloc_keys_address(void **out)
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    static unsigned long long ctx_id[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // 0 before the device's context exists (the lookup below creates it) or when the
    // driver cannot say: the address is then looked up again
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || id == 0 || ctx_id[dev] != id) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_keys);
        if (e != cudaSuccess) return e;
        addr[dev] = ptr;
        ctx_id[dev] = id;
    }
    *out = addr[dev];
    return cudaSuccess;
}

// Sets every key of the allocation-free scratch back to zero (used only after a call
// whose acceptance kernel failed to launch left keys behind).
__global__ void zero_noalloc_keys_kernel()
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < TV_ACCEPT_NOALLOC_MAX_ROWS; i += gridDim.x * blockDim.x)
        g_noalloc_keys[i] = 0ull;
}

cudaError_t launch_accept_noalloc(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                                  const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                                  int32_t *bonus, int32_t *status, int num_sms, cudaStream_t stream)
{
    static std::atomic<uint64_t> dirty{0};  // per device: a failed call may have left keys non-zero
    void *keys = nullptr;
    cudaError_t e = noalloc_keys_address(&keys);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (dirty.load() & bit) {
        zero_noalloc_keys_kernel<<<(TV_ACCEPT_NOALLOC_MAX_ROWS + 255) / 256, 256, 0, stream>>>();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dirty.fetch_and(~bit);
    }
    // the same kernels as tv_accept, on keys that start (and are left) at zero
    e = launch_accept(logits, V, draft, parent, mask, B, nb, am, n_acc, path, bonus, status, keys, num_sms, stream);
    if (e != cudaSuccess) dirty.fetch_or(bit);
    return e;
}

}  // namespace tv
