// a2 + a3 — tree-causal paged attention over a draft tree, with split-KV
// partials merged by a log-sum-exp combine.
//
// What it computes (JETFLOW summary, §2 "Arquitectura Central" tree-causal
// mask and §3 item 3 paged verification attention; DFlash-TfM summary,
// "Declaración del Problema" item 3 ancestor-restricted masking): for every
// sequence b, tree node i and query head h with kv head g = h / G, softmax
// attention of q[b,i,h] over the keys [0, P_b) U {P_b + t : t in anc[i]} of
// the paged cache; O in bf16, LSE = ln sum exp(scaled scores) in fp32.
//
// GB300 design
//   * Work unit ("row tile"): one (sequence, kv head, M tile) with the queries
//     of all G query heads of that kv head packed node-major into 128 rows
//     (row = node_local * G + head_in_group), so each K/V page is read once per
//     (sequence, kv head) and QK^T / PV are 128 x 128 x 128 tcgen05 MMAs.
//   * Stream-K over KV tiles of 128 keys (8 pages): every CTA takes an equal
//     contiguous share of all (row tile, KV tile) pairs, computed in-kernel
//     from prefix_lens (ragged prefixes balance by construction).  A row tile
//     cut between CTAs leaves fp32 partials (normalised O, LSE) in the
//     workspace; each piece then takes a ticket (an epoch-tagged counter per
//     row tile) and the last piece to arrive merges them, so no CTA ever
//     waits for another and no extra launch is needed.
//   * Warp roles per CTA (256 threads): warp 0 issues TMA (Q once per row tile
//     through a 4-D map whose node axis stops at B; K and V one 16-key page x
//     64-column box at a time through a 2-D map over [pages*Hkv*16][D], page ids
//     from the block table, OOB rows zero-filled); warp 1 allocates TMEM and
//     issues tcgen05.mma; warps 4-7 own one TMEM lane = one query row each and
//     run the masked online softmax and the epilogue.
//   * TMEM: two S buffers (128 columns each) so QK^T of tile j+1 overlaps the
//     softmax of tile j, and the O accumulator (128 columns).  P goes to shared
//     memory (bf16, 128-byte swizzled, K-major) and feeds the PV MMA; V is the
//     MN-major B operand.
//   * The ancestor bitmask is read only for KV tiles that reach the tree block
//     [P_b, P_b + B); prefix tiles are unmasked.  The running max is only moved
//     (and O in TMEM rescaled) when a row's max grows by more than 2^8, so the
//     rescale is rare after the first tiles.
//   * Every wait is bounded (tv_device.cuh): a stuck pipeline reports
//     TV_ERR_TIMEOUT and the CTA still frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kM = 128;        // query rows per tile
constexpr int kN = 128;        // keys per KV tile
constexpr int kHeadDim = 128;  // D
constexpr int kPage = 16;      // tokens per KV page
constexpr int kStages = 2;     // K and V ring depth
constexpr int kThreads = 256;
constexpr int kMinTilesPerCta = 2;

constexpr uint32_t kTileBytes = kM * kHeadDim * 2;  // 32 KB: a 128 x 128 bf16 tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;     // one 64-column (128-byte) swizzle column block
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kStages * kTileBytes;
constexpr uint32_t kOffBar = kOffP + 2 * kTileBytes;

enum : int {
    BAR_Q_FULL = 0,
    BAR_Q_EMPTY,
    BAR_K_FULL,                    // + stage
    BAR_K_EMPTY = BAR_K_FULL + 2,  // + stage
    BAR_V_FULL = BAR_K_EMPTY + 2,
    BAR_V_EMPTY = BAR_V_FULL + 2,
    BAR_S_FULL = BAR_V_EMPTY + 2,  // + S buffer
    BAR_P_FULL = BAR_S_FULL + 2,   // + P buffer
    BAR_PV_DONE = BAR_P_FULL + 2,  // + P buffer: PV of that buffer's tile completed
    BAR_O_EMPTY = BAR_PV_DONE + 2,
    BAR_MMA_DONE,
    BAR_COUNT
};
constexpr uint32_t kOffMisc = kOffBar + BAR_COUNT * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1024 bytes

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // S buffer x at column x * 128
constexpr uint32_t kTmemO = 256;  // O accumulator

constexpr uint32_t kIdescQK = umma_idesc_bf16(kM, kN, 0);        // B = K tile, K-major
constexpr uint32_t kIdescPV = umma_idesc_bf16(kM, kHeadDim, 1);  // B = V tile, MN-major
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
    CUtensorMap tm_q;  // 4-D (D, Hq, B, nb), box (64, G, NT, 1)
    CUtensorMap tm_k;  // 2-D (D, num_blocks * Hkv * 16), box (64, 16)
    CUtensorMap tm_v;
    const int32_t *block_table;
    const int32_t *prefix_lens;
    const uint32_t *mask;
    uint16_t *o;
    float *lse;
    int32_t *status;
    float *ws_o;    // [2 * grid][128][128] fp32 partial O (normalised)
    float *ws_lse;  // [2 * grid][128]
    unsigned long long *tickets;  // [nb * Hkv * MT]: (epoch << 32) | pieces that have arrived
    uint32_t epoch;               // distinct for every call
    int nb, B, Hq, Hkv, G, NT, MT, W, max_pages, num_blocks;
    float scale_log2;
};

// ------------------------------------------------------------------ schedule

struct Sched {
    const int32_t *prefix_lens;
    int nb, B, Hkv, NT, MT, max_tokens;
};

__device__ __forceinline__ int rowtile_tiles(int P, int B, int NT, int mt)
{
    const int kv_end = min(B, (mt + 1) * NT);  // tree keys a node of this M tile can see end here
    return (P + kv_end + kN - 1) / kN;
}

// KV tiles of one (sequence, kv head); 0 for a sequence whose prefix does not
// fit its block table (reported as TV_ERR_INVALID_ARG).
__device__ __forceinline__ int head_tiles(const Sched &s, int P)
{
    if (P < 0 || P > s.max_tokens - s.B) return 0;
    int t = 0;
    for (int mt = 0; mt < s.MT; ++mt) t += rowtile_tiles(P, s.B, s.NT, mt);
    return t;
}

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Total (row tile, KV tile) pairs.  Whole warp.
__device__ long long sched_total(const Sched &s, int lane)
{
    long long tot = 0;
    for (int base = 0; base < s.nb; base += 32) {
        const int b = base + lane;
        const long long t = (b < s.nb) ? (long long)s.Hkv * head_tiles(s, __ldg(s.prefix_lens + b)) : 0;
        tot += warp_sum_ll(t);
    }
    return tot;
}

// Sequence and offset inside it of global pair index t (t < total).  Whole warp.
__device__ void sched_locate(const Sched &s, long long t, int lane, int &b_out, long long &off_out)
{
    long long acc = 0;
    for (int base = 0; base < s.nb; base += 32) {
        const int b = base + lane;
        const long long tb = (b < s.nb) ? (long long)s.Hkv * head_tiles(s, __ldg(s.prefix_lens + b)) : 0;
        long long incl = tb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const long long excl = incl - tb;
        const unsigned hit = __ballot_sync(0xffffffffu, tb > 0 && acc + excl <= t && t < acc + incl);
        if (hit) {
            const int l = __ffs(hit) - 1;
            b_out = __shfl_sync(0xffffffffu, b, l);
            off_out = t - acc - __shfl_sync(0xffffffffu, excl, l);
            return;
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    b_out = s.nb;
    off_out = 0;
}

// CTAs that get work: at least kMinTilesPerCta pairs each, at most the grid.
__device__ __forceinline__ long long active_ctas(long long total, int grid)
{
    long long c = (total + kMinTilesPerCta - 1) / kMinTilesPerCta;
    if (c > grid) c = grid;
    return c < 1 ? 1 : c;
}

struct Cursor {
    int b;
    long long off;   // pair offset inside sequence b
    long long left;  // pairs this CTA still has to visit
};

struct Seg {
    int b, g, mt, j0, j1, n_row, P;
};

// Next segment (a run of KV tiles of one row tile) of this CTA's share.
// Row tiles are ordered (sequence, kv head, M tile), KV tiles ascending.
__device__ __forceinline__ bool next_seg(const Sched &s, Cursor &c, Seg &sg)
{
    while (c.left > 0 && c.b < s.nb) {
        const int P = __ldg(s.prefix_lens + c.b);
        const int ht = head_tiles(s, P);
        if (c.off >= (long long)ht * s.Hkv) {
            ++c.b;
            c.off = 0;
            continue;
        }
        const int g = (int)(c.off / ht);
        int rem = (int)(c.off - (long long)g * ht);
        int mt = 0;
        int n = rowtile_tiles(P, s.B, s.NT, 0);
        while (rem >= n) {
            rem -= n;
            ++mt;
            n = rowtile_tiles(P, s.B, s.NT, mt);
        }
        const int take = (int)min((long long)(n - rem), c.left);
        sg.b = c.b;
        sg.g = g;
        sg.mt = mt;
        sg.j0 = rem;
        sg.j1 = rem + take;
        sg.n_row = n;
        sg.P = P;
        c.off += take;
        c.left -= take;
        return true;
    }
    return false;
}

// 32 visibility bits for the keys kstart .. kstart+31 of one query row:
// prefix keys are always visible, tree key P + t iff bit t of the row's mask.
__device__ __forceinline__ uint32_t visible_bits(int kstart, int P, int B, const uint32_t *mrow, int W)
{
    if (kstart + 32 <= P) return 0xffffffffu;
    uint32_t v = (kstart >= P) ? 0u : ((1u << (P - kstart)) - 1u);
    const int t0 = kstart - P;
    if (t0 + 32 > 0 && t0 < B) {
        uint32_t bits;
        if (t0 >= 0) {
            const int w = t0 >> 5, sh = t0 & 31;
            const uint32_t lo = __ldg(mrow + w);
            const uint32_t hi = (w + 1 < W) ? __ldg(mrow + w + 1) : 0u;
            bits = sh ? ((lo >> sh) | (hi << (32 - sh))) : lo;
        } else {
            bits = __ldg(mrow) << (-t0);
        }
        v |= bits;
    }
    return v;
}

// ------------------------------------------------------------------ kernels

__global__ void __launch_bounds__(kThreads, 1) tree_attn_kernel(const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sP = base + kOffP;
    const uint32_t sBar = base + kOffBar;
#define BAR(i) (sBar + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kOffMisc + 4);
    int *sh_b0 = reinterpret_cast<int *>(gbase + kOffMisc + 8);
    long long *sh_off0 = reinterpret_cast<long long *>(gbase + kOffMisc + 16);
    long long *sh_left = reinterpret_cast<long long *>(gbase + kOffMisc + 24);
    long long *sh_total = reinterpret_cast<long long *>(gbase + kOffMisc + 32);
    long long *sh_ctas = reinterpret_cast<long long *>(gbase + kOffMisc + 40);
    long long *sh_t0 = reinterpret_cast<long long *>(gbase + kOffMisc + 48);
    volatile int *sh_last = reinterpret_cast<volatile int *>(gbase + kOffMisc + 56);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Sched sch{p.prefix_lens, p.nb, p.B, p.Hkv, p.NT, p.MT, p.max_pages * kPage};

    if (threadIdx.x == 0) {
        mbar_init(BAR(BAR_Q_FULL), 1);
        mbar_init(BAR(BAR_Q_EMPTY), 1);
        for (int st = 0; st < kStages; ++st) {
            mbar_init(BAR(BAR_K_FULL + st), 1);
            mbar_init(BAR(BAR_K_EMPTY + st), 1);
            mbar_init(BAR(BAR_V_FULL + st), 1);
            mbar_init(BAR(BAR_V_EMPTY + st), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(BAR_S_FULL + x), 1);
            mbar_init(BAR(BAR_P_FULL + x), kM);
            mbar_init(BAR(BAR_PV_DONE + x), 1);
        }
        mbar_init(BAR(BAR_O_EMPTY), kM);
        mbar_init(BAR(BAR_MMA_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2) {
        const long long total = sched_total(sch, lane);
        const long long C = active_ctas(total, gridDim.x);
        const long long c = blockIdx.x;
        long long t0 = 0, t1 = 0;
        if (c < C) {
            t0 = total * c / C;
            t1 = total * (c + 1) / C;
        }
        int b0 = sch.nb;
        long long off0 = 0;
        if (t1 > t0) sched_locate(sch, t0, lane, b0, off0);
        if (lane == 0) {
            *sh_b0 = b0;
            *sh_off0 = off0;
            *sh_left = t1 - t0;
            *sh_total = total;
            *sh_ctas = C;
            *sh_t0 = t0;
        }
        if (blockIdx.x == 0) {
            for (int b = lane; b < sch.nb; b += 32) {
                const int P = __ldg(sch.prefix_lens + b);
                if (P < 0 || P > sch.max_tokens - sch.B) report_status(p.status, TV_ERR_INVALID_ARG);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Cursor cur0{*sh_b0, *sh_off0, *sh_left};

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        Cursor cur = cur0;
        Seg sg;
        uint32_t gt = 0, seg_i = 0;
        bool ok = true;
        const int oob_row = p.num_blocks * p.Hkv * kPage;  // first row past the cache: zero fill
        while (ok && next_seg(sch, cur, sg)) {
            if (seg_i > 0 && !mbar_wait(BAR(BAR_Q_EMPTY), (seg_i - 1) & 1, abort_flag, p.status)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR(BAR_Q_FULL), kTileBytes);
                tma_load_4d(sQ, &p.tm_q, 0, sg.g * p.G, sg.mt * p.NT, sg.b, BAR(BAR_Q_FULL));
                tma_load_4d(sQ + kHalfBytes, &p.tm_q, 64, sg.g * p.G, sg.mt * p.NT, sg.b, BAR(BAR_Q_FULL));
            }
            const int kv_len = sg.P + min(p.B, (sg.mt + 1) * p.NT);
            for (int j = sg.j0; j < sg.j1; ++j, ++gt) {
                const int st = gt & 1;
                const uint32_t ph = (gt >> 1) & 1;
                int row = oob_row;
                if (lane < kN / kPage) {
                    const int pg = j * (kN / kPage) + lane;
                    if (pg * kPage < kv_len) {
                        const int id = __ldg(p.block_table + (size_t)sg.b * p.max_pages + pg);
                        if (id >= 0 && id < p.num_blocks)
                            row = (id * p.Hkv + sg.g) * kPage;
                        else
                            report_status(p.status, TV_ERR_INVALID_ARG);
                    }
                }
                const int my_row = __shfl_sync(0xffffffffu, row, lane >> 1);
                const uint32_t dst_off = (uint32_t)(lane & 1) * kHalfBytes + (uint32_t)(lane >> 1) * (kPage * 128);
                if (!mbar_wait(BAR(BAR_K_EMPTY + st), ph ^ 1, abort_flag, p.status)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(BAR(BAR_K_FULL + st), kTileBytes);
                __syncwarp();
                if (lane < 16) tma_load_2d(sK + st * kTileBytes + dst_off, &p.tm_k, (lane & 1) * 64, my_row, BAR(BAR_K_FULL + st));
                if (!mbar_wait(BAR(BAR_V_EMPTY + st), ph ^ 1, abort_flag, p.status)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(BAR(BAR_V_FULL + st), kTileBytes);
                __syncwarp();
                if (lane < 16) tma_load_2d(sV + st * kTileBytes + dst_off, &p.tm_v, (lane & 1) * 64, my_row, BAR(BAR_V_FULL + st));
            }
            ++seg_i;
        }
        // On an abort, let copies already in flight land before the CTA can exit.
        if (!ok || *abort_flag) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 2000000ull) { }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        Cursor cur = cur0;
        Seg sg;
        uint32_t gt = 0, seg_i = 0;
        bool ok = true;
        auto issue_s = [&](uint32_t t) -> bool {
            const int st = t & 1;
            if (!mbar_wait(BAR(BAR_K_FULL + st), (t >> 1) & 1, abort_flag, p.status)) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t kb = sK + st * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    umma_bf16_ss(tmem + kTmemS + st * 128, sdesc_kmajor_sw128(sQ + off),
                                 sdesc_kmajor_sw128(kb + off), kIdescQK, kk > 0 ? 1u : 0u);
                }
                umma_commit(BAR(BAR_S_FULL + st));
                umma_commit(BAR(BAR_K_EMPTY + st));
            }
            __syncwarp();
            return true;
        };
        while (ok && next_seg(sch, cur, sg)) {
            const int n = sg.j1 - sg.j0;
            if (!mbar_wait(BAR(BAR_Q_FULL), seg_i & 1, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            if (!issue_s(gt)) { ok = false; break; }
            for (int t = 0; t < n; ++t) {
                const uint32_t g_t = gt + t;
                const int buf = g_t & 1;
                if (t + 1 < n && !issue_s(g_t + 1)) { ok = false; break; }
                if (t + 1 == n) {
                    if (lane == 0) umma_commit(BAR(BAR_Q_EMPTY));
                    __syncwarp();
                }
                if (!mbar_wait(BAR(BAR_P_FULL + buf), (g_t >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
                if (t == 0 && seg_i > 0 && !mbar_wait(BAR(BAR_O_EMPTY), (seg_i - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(BAR(BAR_V_FULL + buf), (g_t >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t pb = sP + buf * kTileBytes;
                    const uint32_t vb = sV + buf * kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < kN / 16; ++kk) {
                        umma_bf16_ss(tmem + kTmemO, sdesc_kmajor_sw128(pb + (kk >> 2) * kHalfBytes + (kk & 3) * 32),
                                     sdesc_mnmajor_sw128(vb + kk * 2048, kHalfBytes), kIdescPV,
                                     (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(BAR(BAR_V_EMPTY + buf));
                    umma_commit(BAR(BAR_PV_DONE + buf));
                }
                __syncwarp();
            }
            gt += n;
            ++seg_i;
        }
        // Every MMA this CTA issued completes before TMEM is released.
        if (lane == 0) umma_commit(BAR(BAR_MMA_DONE));
        __syncwarp();
        {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(BAR(BAR_MMA_DONE), 0) && global_timer_ns() - t0 < kWaitLimitNs) { }
        }
    } else if (warp >= 4) {
        // -------------------------------------------------- softmax and epilogue
        const int row = threadIdx.x - 128;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int node_local = row / p.G;
        const int hg = row - node_local * p.G;
        const float sl2 = p.scale_log2;
        const long long total = *sh_total, C = *sh_ctas;
        long long seg_start = *sh_t0;  // global pair index of the current segment's first tile
        Cursor cur = cur0;
        Seg sg;
        uint32_t gt = 0, seg_i = 0;
        bool ok = true;
        while (ok && next_seg(sch, cur, sg)) {
            const int i = sg.mt * p.NT + node_local;
            const bool valid = i < p.B;
            const uint32_t *mrow = p.mask + ((size_t)sg.b * p.B + (valid ? i : 0)) * p.W;
            const int n = sg.j1 - sg.j0;
            float m_run = -INFINITY, l_run = 0.f;  // m_run in log2 units of the scaled score
            for (int t = 0; t < n; ++t) {
                const uint32_t g_t = gt + t;
                const int buf = g_t & 1;
                const int k0 = (sg.j0 + t) * kN;
                if (!mbar_wait(BAR(BAR_S_FULL + buf), (g_t >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + kTmemS + buf * 128 + c * 32, s[c]);
                tmem_ld_wait(s[0]);
                reg_order(s[1]);
                reg_order(s[2]);
                reg_order(s[3]);

                // tree / tail mask (prefix-only tiles skip it), then the row max of the raw scores
                if (!(valid && k0 + kN <= sg.P)) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t vis = valid ? visible_bits(k0 + 32 * c, sg.P, p.B, mrow, p.W) : 0u;
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c][e] = ((vis >> e) & 1u) ? s[c][e] : 0xff800000u;
                    }
                }
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(s[c][e]));
                const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;

                // move the running max only when it grows by more than 2^8
                const float m_new = fmaxf(m_run, tmax);
                if (m_new > m_run + kRescaleLog2) {
                    const float alpha = ex2_approx(m_run - m_new);
                    if (l_run > 0.f) {
                        const uint32_t prev = g_t - 1;
                        if (!mbar_wait(BAR(BAR_PV_DONE + (prev & 1)), (prev >> 1) & 1, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[32];
                            tmem_ld32(lane_addr + kTmemO + c * 32, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(lane_addr + kTmemO + c * 32, o);
                        }
                        tmem_st_wait();
                    }
                    l_run *= alpha;
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;

                // P_j may overwrite its buffer once the PV two tiles back is done
                if (g_t >= 2 &&
                    !mbar_wait(BAR(BAR_PV_DONE + buf), ((g_t - 2) >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t prow = sP + buf * kTileBytes + row * 128;
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const float a = ex2_approx(fmaf(__uint_as_float(s[c][q * 8 + 2 * e2]), sl2, neg_m));
                            const float b = ex2_approx(fmaf(__uint_as_float(s[c][q * 8 + 2 * e2 + 1]), sl2, neg_m));
                            ls[2 * e2] += a;
                            ls[2 * e2 + 1] += b;
                            w[e2] = pack_bf16x2(a, b);
                        }
                        const uint32_t chunk = (uint32_t)((c & 1) * 4 + q);  // 16-byte chunk in the 128-byte row
                        st_shared_v4(prow + (c >> 1) * kHalfBytes + ((chunk ^ (uint32_t)(row & 7)) << 4), w[0], w[1],
                                     w[2], w[3]);
                    }
                }
                l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(BAR(BAR_P_FULL + buf));
            }
            if (!ok) break;
            gt += n;

            // epilogue: O of this row tile is complete once the last PV lands
            const uint32_t last = gt - 1;
            if (!mbar_wait(BAR(BAR_PV_DONE + (last & 1)), (last >> 1) & 1, abort_flag, p.status)) break;
            tc_fence_after();
            uint32_t o[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + kTmemO + c * 32, o[c]);
            tmem_ld_wait(o[0]);
            reg_order(o[1]);
            reg_order(o[2]);
            reg_order(o[3]);
            tc_fence_before();
            mbar_arrive(BAR(BAR_O_EMPTY));

            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const float lse_nat = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            const int h = sg.g * p.G + hg;
            const size_t orow = ((size_t)sg.b * p.B + i) * p.Hq + h;
            uint4 *dst_o = reinterpret_cast<uint4 *>(p.o + orow * kHeadDim);
            if (sg.j0 == 0 && sg.j1 == sg.n_row) {
                if (valid) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[c][q * 8 + 0]) * inv, __uint_as_float(o[c][q * 8 + 1]) * inv);
                            v.y = pack_bf16x2(__uint_as_float(o[c][q * 8 + 2]) * inv, __uint_as_float(o[c][q * 8 + 3]) * inv);
                            v.z = pack_bf16x2(__uint_as_float(o[c][q * 8 + 4]) * inv, __uint_as_float(o[c][q * 8 + 5]) * inv);
                            v.w = pack_bf16x2(__uint_as_float(o[c][q * 8 + 6]) * inv, __uint_as_float(o[c][q * 8 + 7]) * inv);
                            dst_o[c * 4 + q] = v;
                        }
                    }
                    p.lse[orow] = lse_nat;
                }
            } else {
                // A piece of a row tile cut between CTAs c0..c1: park it, take a ticket,
                // and merge all pieces if this one arrived last.
                const long long r0 = seg_start - sg.j0;
                const long long r1 = r0 + sg.n_row;
                const int c0 = (int)(((r0 + 1) * C - 1) / total);
                const int c1 = (int)((r1 * C - 1) / total);
                const size_t slot = 2 * (size_t)blockIdx.x + (seg_i == 0 ? 0 : 1);
                if (valid) {
                    float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (slot * kM + row) * kHeadDim);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[c * 8 + q] = make_float4(
                                __uint_as_float(o[c][q * 4 + 0]) * inv, __uint_as_float(o[c][q * 4 + 1]) * inv,
                                __uint_as_float(o[c][q * 4 + 2]) * inv, __uint_as_float(o[c][q * 4 + 3]) * inv);
                    p.ws_lse[slot * kM + row] = lse_nat;
                }
                __threadfence();
                named_bar_sync(1, kM);
                if (row == 0) {
                    unsigned long long *tk = p.tickets + ((size_t)sg.b * p.Hkv + sg.g) * p.MT + sg.mt;
                    unsigned long long cur_t = *reinterpret_cast<volatile unsigned long long *>(tk);
                    unsigned long long next;
                    for (;;) {
                        next = ((uint32_t)(cur_t >> 32) == p.epoch) ? cur_t + 1
                                                                    : (((unsigned long long)p.epoch << 32) | 1ull);
                        const unsigned long long seen = atomicCAS(tk, cur_t, next);
                        if (seen == cur_t) break;
                        cur_t = seen;
                    }
                    *sh_last = ((int)(next & 0xffffffffull) == c1 - c0 + 1) ? 1 : 0;
                }
                named_bar_sync(1, kM);
                if (*sh_last && valid) {
                    __threadfence();
                    const int slot0 = (r0 == total * c0 / C) ? 2 * c0 : 2 * c0 + 1;
                    float m = -INFINITY;
                    for (int c = c0; c <= c1; ++c)
                        m = fmaxf(m, __ldcg(p.ws_lse + (size_t)(c == c0 ? slot0 : 2 * c) * kM + row));
                    float lse_all = -INFINITY;
                    float wsum = 0.f;
                    if (m != -INFINITY) {
                        for (int c = c0; c <= c1; ++c)
                            wsum += expf(__ldcg(p.ws_lse + (size_t)(c == c0 ? slot0 : 2 * c) * kM + row) - m);
                        lse_all = m + logf(wsum);
                    }
                    for (int part = 0; part < kHeadDim / 32; ++part) {  // 32 output columns at a time
                        float acc[32];
#pragma unroll
                        for (int d = 0; d < 32; ++d) acc[d] = 0.f;
                        if (m != -INFINITY) {
                            for (int c = c0; c <= c1; ++c) {
                                const size_t sl = (size_t)(c == c0 ? slot0 : 2 * c);
                                const float wgt = expf(__ldcg(p.ws_lse + sl * kM + row) - lse_all);
                                const float4 *src =
                                    reinterpret_cast<const float4 *>(p.ws_o + (sl * kM + row) * kHeadDim + part * 32);
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const float4 v = __ldcg(src + q);
                                    acc[4 * q + 0] = fmaf(wgt, v.x, acc[4 * q + 0]);
                                    acc[4 * q + 1] = fmaf(wgt, v.y, acc[4 * q + 1]);
                                    acc[4 * q + 2] = fmaf(wgt, v.z, acc[4 * q + 2]);
                                    acc[4 * q + 3] = fmaf(wgt, v.w, acc[4 * q + 3]);
                                }
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack_bf16x2(acc[8 * q + 0], acc[8 * q + 1]);
                            v.y = pack_bf16x2(acc[8 * q + 2], acc[8 * q + 3]);
                            v.z = pack_bf16x2(acc[8 * q + 4], acc[8 * q + 5]);
                            v.w = pack_bf16x2(acc[8 * q + 6], acc[8 * q + 7]);
                            dst_o[part * 4 + q] = v;
                        }
                    }
                    p.lse[orow] = lse_all;
                }
            }
            seg_start += n;
            ++seg_i;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
#undef BAR
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

size_t attn_workspace_bytes(int ctas, int row_tiles)
{
    return (size_t)2 * ctas * kM * (kHeadDim + 1) * sizeof(float) + (size_t)row_tiles * sizeof(unsigned long long);
}

int attn_row_tiles(const tv_attn_args *a)
{
    const int NT = kM / (a->Hq / a->Hkv);
    return a->nb * a->Hkv * ((a->B + NT - 1) / NT);
}

// Every call gets its own ticket epoch, so tickets left by an earlier (even an
// interrupted) call never count towards this one.
static uint32_t next_epoch()
{
    static std::atomic<uint32_t> counter{0};
    uint32_t e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    if (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    return e;
}

int32_t launch_attn(const tv_attn_args *a, int ctas, void *workspace, cudaStream_t stream, cudaError_t *cuda_err)
{
    *cuda_err = cudaSuccess;
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        *cuda_err = cudaErrorNotSupported;
        return TV_ERR_CUDA;
    }
    AttnParams p;
    memset(&p, 0, sizeof(p));
    const int G = a->Hq / a->Hkv;
    const int NT = kM / G;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)a->Hq, (cuuint64_t)a->B, (cuuint64_t)a->nb};
        const cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)a->Hq * kHeadDim * 2,
                                       (cuuint64_t)a->B * a->Hq * kHeadDim * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)NT, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a->q_d), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *cuda_err = cudaErrorInvalidValue;
            return TV_ERR_CUDA;
        }
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)a->num_blocks * a->Hkv * kPage};
        const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)kPage};
        const cuuint32_t es[2] = {1, 1};
        for (int which = 0; which < 2; ++which) {
            CUtensorMap *tm = which ? &p.tm_v : &p.tm_k;
            void *ptr = const_cast<void *>(which ? a->v_cache_d : a->k_cache_d);
            if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
                *cuda_err = cudaErrorInvalidValue;
                return TV_ERR_CUDA;
            }
        }
    }
    p.block_table = a->block_table_d;
    p.prefix_lens = a->prefix_lens_d;
    p.mask = a->mask_d;
    p.o = static_cast<uint16_t *>(a->o_d);
    p.lse = a->lse_d;
    p.status = a->dev_status_d;
    p.ws_o = static_cast<float *>(workspace);
    p.ws_lse = p.ws_o + (size_t)2 * ctas * kM * kHeadDim;
    p.tickets = reinterpret_cast<unsigned long long *>(p.ws_lse + (size_t)2 * ctas * kM);
    p.epoch = next_epoch();
    p.nb = a->nb;
    p.B = a->B;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.G = G;
    p.NT = NT;
    p.MT = (a->B + NT - 1) / NT;
    p.W = (a->B + 31) / 32;
    p.max_pages = a->max_pages;
    p.num_blocks = a->num_blocks;
    const float scale = a->scale > 0.f ? a->scale : 1.0f / sqrtf((float)kHeadDim);
    p.scale_log2 = scale * 1.4426950408889634f;

    cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) {
        tree_attn_kernel<<<ctas, kThreads, kSmemBytes, stream>>>(p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        *cuda_err = e;
        return TV_ERR_CUDA;
    }
    return TV_OK;
}

}  // namespace tv
