// Rollback-free tree verification through a Gated DeltaNet layer.
//
// DFlash-TfM summary, §3 "Verificación de Árboles sin Rollback": the state follows
//   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
// the tree is topologically ordered, the verification is a masked triangular solve
// (I + X) U = beta V over the tree, and the committed state is not touched.  Every
// node's output is o_i = S_i^T q_i for the state its own root path builds from S0.
// With gamma_i the product of alpha over i's root path (i included) and
// r_ij = gamma_i / gamma_j, that state is S_i = gamma_i S0 + sum_{j in path(i)}
// r_ij k_j u_j^T, where
//   u_i = beta_i (v_i - gamma_i S0^T k_i) - sum_{j strict ancestor} beta_i r_ij (k_i . k_j) u_j
//   o_i = gamma_i S0^T q_i + sum_{j in path(i)} r_ij (q_i . k_j) u_j.
// (X_ij = beta_i r_ij k_i.k_j and Y_ij = r_ij q_i.k_j are the pages' interaction
// matrices, restricted to ancestors by the tree mask.)
//
// GPU form: one fused kernel, 16 warps per CTA.  The value columns are split: u_i
// and o_i restricted to a set of value columns need only those columns of S0 and
// v_i (the Gram entries and decays are shared by all columns), so each (sequence,
// head) runs as 4 CTAs of 32 value columns each, every one doing the whole tree
// for its columns (the Gram part is recomputed per CTA: it is the cheap part).
//   1. Stage, with every global load issued at once: the K and Q rows (cp.async)
//      as K-major 128-byte-swizzled bf16 tiles, the slice's v columns (B <= 128),
//      the slice of S0 (through registers, split into bf16 hi + lo parts, S0 = hi +
//      lo to ~2^-17, transposed into one K-major swizzled 64-row tile), the parent
//      array (validated), and a walk up each node's root path that sets its
//      ancestor bits and writes, per ancestor j (slot = distance to i - 1), the
//      record (j, r_ij): r_ij is the running product of the alphas passed, and
//      gamma_i the product over the whole path.
//   2. Tensor cores (tcgen05, fp32 accumulators in TMEM): the Gram blocks K K^T and
//      Q K^T (committed first, so the epilogue starts on them early), then the
//      slice's K S0 and Q S0 (N = 64: the hi and lo parts side by side, added in the
//      epilogue, so fp32-accurate), 128 nodes per M tile (two tiles and three passes
//      for B > 128).
//   3. Epilogue, all warps (warp w reads TMEM lanes 32 (w % 4).. and columns
//      32 (w / 4)..): for each ancestor j of i (its bit in i's mask; its slot is the
//      count of mask bits above it), the pair (k_i.k_j, q_i.k_j) into j's record
//      (the first 24 records of a node in shared memory when B <= 128, the rest in
//      the workspace); the first four warps also form the slice of
//      r_i = beta_i (v_i - gamma_i (K S0)_i) and o0_i = gamma_i (Q S0)_i.
//   4. Solve, warp per node in dataflow order, one value column per lane: node i's
//      r_i and o0_i rows are loaded (the warp's next node's while this one runs);
//      node i waits (bounded, asleep on an mbarrier) for its grandparent's u row and
//      adds the terms of every ancestor above its parent (each one broadcast record
//      load, one u-row load and two fused multiply-adds, four ancestors in flight),
//      then waits for its parent's row and adds that term alone, so the chain down
//      the tree costs one term per level.  Warps take nodes in index order, so the
//      smallest unfinished node can always run: every wait ends.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kGdnD = 128;
constexpr int kGdnMaxB = 256;
constexpr int kGdnThreads = 512;
constexpr int kGdnWarps = kGdnThreads / 32;
constexpr uint32_t kGdnTile = 128 * 128 * 2;  // one 128 x 128 bf16 operand tile
constexpr uint32_t kGdnHalf = kGdnTile / 2;   // one 64-column (128-byte) swizzle block of it
constexpr int kGdnMaskWords = kGdnMaxB / 32;
constexpr int kGdnSlices = 4;                      // CTAs per (sequence, head), one per value-column slice
constexpr int kGdnCols = kGdnD / kGdnSlices;       // 32 value columns per CTA: one per lane in the solve
constexpr uint32_t kGdnRowBytes = kGdnCols * 4;    // an fp32 row slice (r, u, o0)
// The S0 slice as one B operand, transposed and K-major: rows 0..31 its hi part, rows
// 32..63 its lo part (value column n in rows n and 32 + n), 128 keys per row, bf16
constexpr uint32_t kGdnSTile = 2 * kGdnCols * kGdnD * 2;
constexpr uint32_t kGdnSHalf = kGdnSTile / 2;  // its 64-key (128-byte) swizzle column block
static_assert(kGdnCols == 32, "one value column per lane");
constexpr int kGdnSmemSlots = 24;             // records per node kept in shared memory (B <= 128)
constexpr uint32_t kGdnTmemCols = 512;
// TMEM columns of one pass: K S0, Q S0 (32 each), then the K K^T and Q K^T blocks
constexpr uint32_t kColKS = 0, kColQS = 128, kColKK = 256, kColQK = 384;
constexpr uint32_t kIdescS = umma_idesc_bf16(128, 2 * kGdnCols, 0);  // B = the S0 slice's hi and lo rows
constexpr uint32_t kIdescG = umma_idesc_bf16(128, 128, 0);  // B = K tile, K-major

// One ancestor j of a node i: its index, the decay ratio r_ij (written by the root
// walk) and the two Gram entries k_i.k_j, q_i.k_j (written by the epilogue).
struct __align__(16) GdnRec {
    int32_t j;
    float r, kk, qk;
};

struct GdnSmem {
    uint32_t k, q, s, tiles_end;
    uint32_t recs, v;  // B <= 128 only: records [kGdnSmemSlots][128] (slot-major), v rows [128][32 columns] bf16
    uint32_t done, parent, alpha, beta, gamma, depth, yii, mask, total;
};

__host__ __device__ inline GdnSmem gdn_smem_layout(int B)
{
    GdnSmem L;
    const uint32_t T = (uint32_t)(B + 127) / 128;
    L.k = 0;
    L.q = T * kGdnTile;
    L.s = 2 * T * kGdnTile;
    L.tiles_end = L.s + kGdnSTile;
    uint32_t o = L.tiles_end;
    L.recs = L.v = 0;
    if (B <= 128) {
        L.recs = o;
        o += 128u * kGdnSmemSlots * 16u;
        L.v = o;
        o += 128u * kGdnCols * 2u;
    }
    const uint32_t a = 4u * (uint32_t)B;
    L.done = o; o += 2 * a;  // one mbarrier per node
    L.parent = o; o += a;
    L.alpha = o; o += a;
    L.beta = o; o += a;
    L.gamma = o; o += a;
    L.depth = o; o += a;
    L.yii = o; o += a;
    L.mask = o; o += 4u * kGdnMaskWords * (uint32_t)B;
    L.total = o;
    return L;
}

// byte offset of column c (0..31) of the fp32 row slice of node i: 16-byte chunks
// swizzled by (i & 7), so a warp's one-row reads and its 32-row chunk writes are
// both free of bank conflicts
__device__ __forceinline__ uint32_t row_col(int i, int c)
{
    return (uint32_t)i * kGdnRowBytes + ((((uint32_t)c >> 2) ^ ((uint32_t)i & 7u)) << 4) + ((uint32_t)c & 3u) * 4u;
}

// round-to-nearest bf16 bits of x
__device__ __forceinline__ uint32_t bf16_bits(float x)
{
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

// 16-byte global -> shared copy, zero-filled when !valid (nothing is read then)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// record slot `slot` of node i: the first kGdnSmemSlots in shared memory when B <= 128,
// slot-major there (the threads of a warp, one node each, write one slot side by side,
// free of bank conflicts), node-major in the workspace
__device__ __forceinline__ GdnRec *rec_at(GdnRec *s_recs, GdnRec *g_recs, bool small, int B, int i, int slot)
{
    return (small && slot < kGdnSmemSlots) ? s_recs + slot * 128 + i : g_recs + (size_t)i * B + slot;
}

__global__ void __launch_bounds__(kGdnThreads, 1) gdn_tree_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const float *__restrict__ alpha, const float *__restrict__ beta, const float *__restrict__ S0,
    const int32_t *__restrict__ parent, int B, int H, float *__restrict__ O, void *__restrict__ ws, int32_t *status)
{
    extern __shared__ uint8_t gdn_raw[];
    __shared__ __align__(8) uint64_t s_bar[2];  // Gram MMAs done, S0 MMAs done
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const uint32_t raw = smem_u32(gdn_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gb = gdn_raw + (base - raw);
    const GdnSmem L = gdn_smem_layout(B);
    int *s_parent = reinterpret_cast<int *>(gb + L.parent);
    float *s_alpha = reinterpret_cast<float *>(gb + L.alpha);
    float *s_beta = reinterpret_cast<float *>(gb + L.beta);
    float *s_gamma = reinterpret_cast<float *>(gb + L.gamma);
    int *s_depth = reinterpret_cast<int *>(gb + L.depth);
    float *s_yii = reinterpret_cast<float *>(gb + L.yii);
    const uint32_t done_bar = base + L.done;  // node i's mbarrier at done_bar + 8 i: phase 0 completes when u_i is written
    uint32_t *s_mask = reinterpret_cast<uint32_t *>(gb + L.mask);  // word w of node i at [w * B + i]

    const int h = blockIdx.x, b = blockIdx.y, nb = gridDim.y;
    const int c0 = blockIdx.z * kGdnCols;  // this CTA's value columns c0 .. c0 + 31
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = (B + 127) >> 7;
    const bool small = B <= 128;  // one M tile: r / u and o0 rows, records and v rows fit in shared memory
    const size_t bh = (size_t)b * H + h, bhs = bh * kGdnSlices + blockIdx.z;
    // workspace, per (sequence, head, slice): records [B][B]; for B > 128 also r and o0
    // row slices [B][32] each
    GdnRec *g_recs = reinterpret_cast<GdnRec *>(ws) + bhs * B * B;
    GdnRec *s_recs = reinterpret_cast<GdnRec *>(gb + L.recs);
    float *g_rows = reinterpret_cast<float *>(reinterpret_cast<GdnRec *>(ws) + (size_t)nb * H * kGdnSlices * B * B);
    uint8_t *r_rows = small ? gb : reinterpret_cast<uint8_t *>(g_rows + bhs * B * kGdnCols);
    uint8_t *o0_rows = small ? gb + 128 * kGdnRowBytes
                             : reinterpret_cast<uint8_t *>(g_rows + ((size_t)nb * H * kGdnSlices + bhs) * B * kGdnCols);
    const uint32_t bar_g = smem_u32(&s_bar[0]), bar_s = smem_u32(&s_bar[1]);

    pdl_wait_primary();  // every input may come from the previous kernel
    pdl_launch_dependents();

    // ---- every global load at once: the tree first, then K, Q (and v) rows by cp.async
    // and S0 into registers
    int pv[2] = {0, 0};
    float av[2] = {0.f, 0.f}, bv[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int i = tid + e * kGdnThreads;
        if (i < B) {
            const size_t row = ((size_t)b * B + i) * H + h;
            pv[e] = parent[(size_t)b * B + i];
            av[e] = alpha[row];
            bv[e] = beta[row];
        }
    }
    const int n16 = T * 128 * 16;  // 16-byte chunks per operand tile set
    for (int idx = tid; idx < 2 * n16; idx += kGdnThreads) {
        const int which = idx >= n16, r = idx - which * n16, i = r >> 4, c = r & 15;
        const uint32_t dst = base + (which ? L.q : L.k) + (uint32_t)(i >> 7) * kGdnTile + (uint32_t)(c >> 3) * kGdnHalf +
                             (uint32_t)(i & 127) * 128 + ((uint32_t)((c & 7) ^ (i & 7)) << 4);
        const uint16_t *src = (which ? q : k) + (((size_t)b * B + min(i, B - 1)) * H + h) * kGdnD + c * 8;
        cp_async16(dst, src, i < B);
    }
    if (small) {  // the slice's v columns [i][4 chunks], chunks swizzled by (i & 3)
        for (int idx = tid; idx < B * 4; idx += kGdnThreads) {
            const int i = idx >> 2, c = idx & 3;
            cp_async16(base + L.v + (uint32_t)i * 64 + ((uint32_t)(c ^ (i & 3)) << 4),
                       v + (((size_t)b * B + i) * H + h) * kGdnD + c0 + c * 8, true);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // the S0 slice: warp w, lane l holds value column c0 + l for keys 8 w .. 8 w + 7
    static_assert(kGdnWarps * 8 == kGdnD, "S0 slice split");
    float sv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sv[e] = S0[(bh * kGdnD + 8 * warp + e) * kGdnD + c0 + lane];

    bool bad = false;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int i = tid + e * kGdnThreads;
        if (i < B) {
            bad |= (i == 0) ? (pv[e] != -1) : (pv[e] < 0 || pv[e] >= i);
            s_parent[i] = pv[e];
            s_alpha[i] = av[e];
            s_beta[i] = bv[e];
            mbar_init(done_bar + 8u * (uint32_t)i, 32);  // one arrival per lane of the solving warp
        }
    }
    if (tid == 0) {
        s_abort = 0;
        mbar_init(bar_g, 1);
        mbar_init(bar_s, 1);
    }
    fence_mbar_init();
    if (__syncthreads_or(bad)) {
        cp_async_wait_all();
        if (tid == 0) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
        return;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kGdnTmemCols);
        tmem_relinquish();
    }

    // root paths: ancestor bits, records (j, r_ij) in slot order, depth and gamma
    for (int i = tid; i < B; i += kGdnThreads) {
        uint32_t *m = s_mask + i;  // word w at m[w * B]: the threads of a warp touch consecutive words
#pragma unroll
        for (int w = 0; w < kGdnMaskWords; ++w) m[w * B] = 0;  // all 8 words (zeros past B)
        m[(i >> 5) * B] = 1u << (i & 31);
        float r = s_alpha[i];
        int slot = 0;
        for (int j = s_parent[i]; j >= 0; j = s_parent[j], ++slot) {
            m[(j >> 5) * B] |= 1u << (j & 31);
            GdnRec *rc = rec_at(s_recs, g_recs, small, B, i, slot);
            rc->j = j;
            rc->r = r;
            r *= s_alpha[j];
        }
        s_depth[i] = slot;
        s_gamma[i] = r;
    }
    // the S0 slice [key r][value c0 + n] -> hi and lo bf16 parts, transposed: row n
    // holds keys 0..127 (K-major, 128-byte swizzled, like the K and Q tiles)
    // (keys 8 w .. 8 w + 7 of row n are one 16-byte chunk: one store per part)
    {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            hi[e] = bf16_bits(sv[e]);
            lo[e] = bf16_bits(sv[e] - __uint_as_float(hi[e] << 16));
        }
        const int n = lane, r0 = 8 * warp;  // row n: hi; row 32 + n: lo (same swizzle: 32 is a multiple of 8)
        const uint32_t off =
            (uint32_t)(r0 >> 6) * kGdnSHalf + (uint32_t)n * 128 + ((uint32_t)(((r0 & 63) >> 3) ^ (n & 7)) << 4);
        st_shared_v4(base + L.s + off, hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16), hi[4] | (hi[5] << 16),
                     hi[6] | (hi[7] << 16));
        st_shared_v4(base + L.s + off + kGdnCols * 128, lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16),
                     lo[4] | (lo[5] << 16), lo[6] | (lo[7] << 16));
    }
    cp_async_wait_all();
    fence_proxy_async_smem();  // the tensor core reads what these threads wrote
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // ---- passes: (M tile m, with K S0 / Q S0?, Gram column block n)
    const int npass = T == 1 ? 1 : 3;
    const int quarter = warp & 3, chunk = warp >> 2;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * quarter) << 16);
    for (int p = 0; p < npass; ++p) {
        const int m = p == 0 ? 0 : 1, n = p == 2 ? 1 : 0;
        const bool has_s = p < 2;
        if (tid == 0) {
            const uint32_t kA = base + L.k + (uint32_t)m * kGdnTile, qA = base + L.q + (uint32_t)m * kGdnTile;
            const uint32_t kB = base + L.k + (uint32_t)n * kGdnTile;
#pragma unroll
            for (int kk = 0; kk < kGdnD / 16; ++kk) {
                const uint32_t off = (uint32_t)(kk >> 2) * kGdnHalf + (uint32_t)(kk & 3) * 32;
                const uint32_t acc = kk > 0 ? 1u : 0u;
                umma_bf16_ss(tmem + kColKK, sdesc_kmajor_sw128(kA + off), sdesc_kmajor_sw128(kB + off), kIdescG, acc);
                umma_bf16_ss(tmem + kColQK, sdesc_kmajor_sw128(qA + off), sdesc_kmajor_sw128(kB + off), kIdescG, acc);
            }
            umma_commit(bar_g);
            if (has_s) {
#pragma unroll
                for (int kk = 0; kk < kGdnD / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kGdnHalf + (uint32_t)(kk & 3) * 32;
                    const uint32_t acc = kk > 0 ? 1u : 0u;
                    const uint64_t sd =
                        sdesc_kmajor_sw128(base + L.s + (uint32_t)(kk >> 2) * kGdnSHalf + (uint32_t)(kk & 3) * 32);
                    umma_bf16_ss(tmem + kColKS, sdesc_kmajor_sw128(kA + off), sd, kIdescS, acc);
                    umma_bf16_ss(tmem + kColQS, sdesc_kmajor_sw128(qA + off), sd, kIdescS, acc);
                }
                umma_commit(bar_s);
            }
        }
        const int i = 128 * m + 32 * quarter + lane;  // this thread's TMEM lane = node
        const bool live = i < B;
        const bool s_warp = has_s && chunk == 0;  // the first four warps form the r and o0 row slices
        uint4 vv[4];
        if (s_warp && live) {
            if (small) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    vv[e] = *reinterpret_cast<const uint4 *>(gb + L.v + i * 64 + ((e ^ (i & 3)) << 4));
            } else {
                const uint4 *vr = reinterpret_cast<const uint4 *>(v + (((size_t)b * B + i) * H + h) * kGdnD + c0);
#pragma unroll
                for (int e = 0; e < 4; ++e) vv[e] = vr[e];
            }
        }
        // Gram entries of node i's ancestors j = 128 n + 32 chunk + t (and of i itself)
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar_g, (uint32_t)(p & 1), &s_abort, status));
        if (ok) {
            tc_fence_after();
            uint32_t x[32], y[32];
            tmem_ld32(t_lane + kColKK + 32 * chunk, x);
            tmem_ld32(t_lane + kColQK + 32 * chunk, y);
            tmem_ld_wait(x);
            reg_order(y);
            if (live) {
                // node i's bits are its ancestors and itself (its highest bit), so ancestor j's
                // slot (0 = the parent) is the number of bits above j, minus one
                const int w = 4 * n + chunk;
                const uint32_t bits = s_mask[w * B + i];
                int above = -1;
#pragma unroll
                for (int ww = 0; ww < kGdnMaskWords; ++ww)
                    if (ww > w) above += __popc(s_mask[ww * B + i]);
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    if ((bits >> t) & 1u) {
                        const int j = 32 * w + t;
                        if (j == i) {
                            s_yii[i] = __uint_as_float(y[t]);
                        } else {
                            const int slot = above + __popc(t == 31 ? 0u : bits >> (t + 1));
                            GdnRec *rc = rec_at(s_recs, g_recs, small, B, i, slot);
                            rc->kk = __uint_as_float(x[t]);
                            rc->qk = __uint_as_float(y[t]);
                        }
                    }
                }
            }
        }
        if (ok && has_s) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar_s, (uint32_t)(p & 1), &s_abort, status));
            if (ok && s_warp) {
                tc_fence_after();
                uint32_t x[32], y[32], xl[32];
                // (K S0)_i = K hi + K lo: the two halves of the 64 accumulator columns
                tmem_ld32(t_lane + kColKS, x);
                tmem_ld32(t_lane + kColKS + kGdnCols, xl);
                tmem_ld_wait(x);
                reg_order(xl);
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) + __uint_as_float(xl[c]));
                tmem_ld32(t_lane + kColQS, y);
                tmem_ld32(t_lane + kColQS + kGdnCols, xl);
                tmem_ld_wait(y);
                reg_order(xl);
#pragma unroll
                for (int c = 0; c < 32; ++c) y[c] = __float_as_uint(__uint_as_float(y[c]) + __uint_as_float(xl[c]));
                if (live) {
                    const float bi = s_beta[i], gi = s_gamma[i];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {  // 16-byte chunk e: slice columns 4 e ..
                        const uint4 w = vv[e >> 1];
                        const uint32_t w0 = (e & 1) ? w.z : w.x, w1 = (e & 1) ? w.w : w.y;
                        const float vx[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
                        float4 r4, o4;
                        r4.x = bi * (vx[0] - gi * __uint_as_float(x[4 * e + 0]));
                        r4.y = bi * (vx[1] - gi * __uint_as_float(x[4 * e + 1]));
                        r4.z = bi * (vx[2] - gi * __uint_as_float(x[4 * e + 2]));
                        r4.w = bi * (vx[3] - gi * __uint_as_float(x[4 * e + 3]));
                        o4.x = gi * __uint_as_float(y[4 * e + 0]);
                        o4.y = gi * __uint_as_float(y[4 * e + 1]);
                        o4.z = gi * __uint_as_float(y[4 * e + 2]);
                        o4.w = gi * __uint_as_float(y[4 * e + 3]);
                        const uint32_t off = row_col(i, 4 * e);
                        *reinterpret_cast<float4 *>(r_rows + off) = r4;  // over the finished tiles when small
                        *reinterpret_cast<float4 *>(o0_rows + off) = o4;
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (s_abort) break;
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kGdnTmemCols);
    }
    if (s_abort) return;

    // ---- solve: warp per node, in index order, lane = value column; the next node's
    // rows load during this one
    uint8_t *s_u = gb;  // u row slices (fp32, swizzled 16-byte chunks) over the finished operand tiles
    float r_n = 0.f, o_n = 0.f;
    if (warp < B) {
        r_n = *reinterpret_cast<const float *>(r_rows + row_col(warp, lane));
        o_n = *reinterpret_cast<const float *>(o0_rows + row_col(warp, lane));
    }
    for (int i = warp; i < B; i += kGdnWarps) {
        const int p = s_parent[i], di = s_depth[i];
        const float bi = s_beta[i], yii = s_yii[i];
        float u = r_n, o = o_n;
        if (i + kGdnWarps < B) {
            r_n = *reinterpret_cast<const float *>(r_rows + row_col(i + kGdnWarps, lane));
            o_n = *reinterpret_cast<const float *>(o0_rows + row_col(i + kGdnWarps, lane));
        }
        // Ancestor terms in slot order from slot l0 on, up to slot l1: four in flight at a time
        // (records from shared memory), or, for deep paths, 32 records at a time, one per
        // lane, then broadcast.
        auto accumulate = [&](int l0, int l1) {
            if (small && l1 <= kGdnSmemSlots) {
                const GdnRec *recs_i = s_recs + i;  // slot l at recs_i[128 l]
                for (int l = l0; l < l1; l += 4) {
                    GdnRec rc[4];
                    float uj[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (l + e < l1) rc[e] = recs_i[128 * (l + e)];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (l + e < l1) uj[e] = *reinterpret_cast<const float *>(s_u + row_col(rc[e].j, lane));
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (l + e < l1) {
                            u -= bi * rc[e].r * rc[e].kk * uj[e];
                            o += rc[e].r * rc[e].qk * uj[e];
                        }
                }
                return;
            }
            for (int lb = l0; lb < l1; lb += 32) {
                const int n = min(l1 - lb, 32);
                GdnRec mine = {0, 0.f, 0.f, 0.f};
                if (lane < n) mine = *rec_at(s_recs, g_recs, small, B, i, lb + lane);
                const float xm = bi * mine.r * mine.kk, ym = mine.r * mine.qk;
                for (int e0 = 0; e0 < n; e0 += 4) {
                    int jj[4];
                    float xx[4], yy[4], uj[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        jj[e] = __shfl_sync(0xffffffffu, mine.j, e0 + e);
                        xx[e] = __shfl_sync(0xffffffffu, xm, e0 + e);
                        yy[e] = __shfl_sync(0xffffffffu, ym, e0 + e);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (e0 + e < n) uj[e] = *reinterpret_cast<const float *>(s_u + row_col(jj[e], lane));
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (e0 + e < n) {
                            u -= xx[e] * uj[e];
                            o += yy[e] * uj[e];
                        }
                }
            }
        };
        // Wait (bounded; the hardware suspends the warp) until the grandparent's u row is
        // written: then every ancestor's above the parent is, and the acquire makes them
        // visible, so their terms are added while the parent is still being solved.  Then
        // wait for the parent and add its term: only that one is on the chain down the tree.
        const int gp = p >= 0 ? s_parent[p] : -1;
        if (gp >= 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(done_bar + 8u * (uint32_t)gp, 0, &s_abort, status))) break;
            accumulate(1, di);
        }
        if (p >= 0) {  // slot 0 is the parent: its record is read before the wait, its row after
            const GdnRec rp = *rec_at(s_recs, g_recs, small, B, i, 0);
            if (!__all_sync(0xffffffffu, mbar_wait(done_bar + 8u * (uint32_t)p, 0, &s_abort, status))) break;
            const float up = *reinterpret_cast<const float *>(s_u + row_col(p, lane));
            u -= bi * rp.r * rp.kk * up;
            o += rp.r * rp.qk * up;
        }
        // every lane arrives (the barrier counts 32): each arrival releases that lane's
        // part of u_i, so the phase completes once the whole row is written
        *reinterpret_cast<float *>(s_u + row_col(i, lane)) = u;
        mbar_arrive(done_bar + 8u * (uint32_t)i);
        o += yii * u;
        O[(((size_t)b * B + i) * H + h) * kGdnD + c0 + lane] = o;
    }
}

size_t gdn_workspace_bytes(int nb, int B, int H)
{
    size_t bytes = (size_t)nb * H * kGdnSlices * B * B * sizeof(GdnRec);
    if (B > 128) bytes += (size_t)2 * nb * H * kGdnSlices * B * kGdnCols * sizeof(float);
    return bytes;
}

cudaError_t launch_gdn_tree(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                            const float *beta, const float *S0, const int32_t *parent, int nb, int B, int H, float *O,
                            void *workspace, int32_t *status, cudaStream_t stream)
{
    static int opted_in[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(dev >= 0 && dev < 64 && opted_in[dev])) {
        const uint32_t most = gdn_smem_layout(128).total > gdn_smem_layout(kGdnMaxB).total
                                  ? gdn_smem_layout(128).total
                                  : gdn_smem_layout(kGdnMaxB).total;  // the largest layout over 1 <= B <= 256
        e = cudaFuncSetAttribute(gdn_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(most + 1024));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = 1;
    }
    return launch_dependent(gdn_tree_kernel, dim3((unsigned)H, (unsigned)nb, (unsigned)kGdnSlices), dim3(kGdnThreads),
                            gdn_smem_layout(B).total + 1024, stream, q, k, v, alpha, beta, S0, parent, B, H, O,
                            workspace, status);
}

}  // namespace tv
