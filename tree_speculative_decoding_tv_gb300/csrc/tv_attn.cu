// Tree-causal paged attention over a draft tree, with split-KV
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
//   * Rows: the queries of all G query heads of one kv head are packed
//     node-major into 128-row M tiles (row = node_local * G + head_in_group),
//     so each K/V page is read once per (sequence, kv head).  A CTA works on a
//     PAIR of M tiles (A = 2mp, B = 2mp + 1) of the same (sequence, kv head):
//     every K/V tile it loads feeds both, halving K/V traffic per MMA.
//   * Stream-K: the (pair tile, 128-key KV tile) items of all sequences are
//     cut into equal contiguous shares, one per CTA, computed in-kernel from
//     prefix_lens, so ragged prefixes balance by construction.  A pair tile cut
//     between CTAs leaves partials (normalised O in fp16, LSE) in the
//     workspace.  When the cut tiles have few pieces, each 32-row quarter of a
//     tile counts its pieces in and the warp whose piece lands last merges that
//     quarter right away; otherwise a merge kernel launched as a programmatic
//     dependent of this one combines them with every SM at once.  No CTA ever
//     waits on another.
//   * Warp roles (384 threads): warp 0 issues TMA (Q by a 4-D map whose node
//     axis stops at B; K/V one 16-key page x 64 columns per copy through a 2-D
//     map over [pages*Hkv*16][D], page ids from the block table, rows past the
//     needed keys zero-filled; evict-first in L2 when no other CTA reads them); warp 1 owns TMEM and issues tcgen05.mma;
//     warpgroups 1 and 2 run the softmax of tiles A and B, one TMEM lane (one
//     query row) per thread.  setmaxnreg moves registers from warpgroup 0 to
//     the softmax warpgroups.
//   * TMEM (512 columns): S_A, O_A, S_B, O_B, 128 columns each.  The softmax
//     writes P (bf16) back over the first 64 columns of its S and the PV MMA
//     reads A = P straight from TMEM; V is the MN-major B operand in shared
//     memory.  Issue order per KV tile j: PV_A(j), QK_A(j+1), PV_B(j),
//     QK_B(j+1), so each softmax warpgroup works while the tensor core runs the
//     other tile's two MMAs.
//   * A pair whose second M tile does not exist (B rows fit one tile) runs in
//     single-tile mode: both softmax warpgroups serve M tile A, warpgroup x
//     taking the KV tiles with index % 2 == x into S_x / O_x, and warpgroup A
//     combines the two halves (O_A, O_B read straight from TMEM) at the end, so
//     softmax and MMAs still overlap.
//   * The ancestor bitmask is read only for KV tiles that reach the tree block
//     [P_b, P_b + B); prefix tiles are unmasked.  A row's running max only
//     moves (and O in TMEM is rescaled) when it grows by more than 2^8.  The
//     commit behind S(j) also covers PV(j-1), so that rescale needs no wait.
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

constexpr int kM = 128;        // query rows per M tile
constexpr int kN = 128;        // keys per KV tile
constexpr int kHeadDim = 128;  // D
constexpr int kPage = 16;      // tokens per KV page
constexpr int kSlots = 5;      // K/V ring: K(j) -> slot (2j) % 5, V(j) -> slot (2j + 1) % 5
constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = kM / 32;  // warps of one softmax warpgroup: each arrives once per phase
constexpr int kMinTilesPerCta = 2;
constexpr int kAlignedMaxTiles = 8;  // unit-aligned schedule: at most this many KV tiles per unit
constexpr uint32_t kRegsLow = 64;    // warpgroup 0 after setmaxnreg.dec (128 x 64 + 256 x 216 <= 384 x 168)
constexpr uint32_t kRegsHigh = 216; // softmax warpgroups after setmaxnreg.inc

constexpr uint32_t kTileBytes = kM * kHeadDim * 2;  // 32 KB: a 128 x 128 bf16 tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;     // one 64-column (128-byte) swizzle column block
constexpr uint32_t kOffQ = 0;                       // Q_A, Q_B
constexpr uint32_t kOffKV = kOffQ + 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffKV + kSlots * kTileBytes;

enum : int {
    BAR_Q_FULL = 0,
    BAR_Q_EMPTY,
    BAR_KV_FULL,                         // + slot
    BAR_KV_EMPTY = BAR_KV_FULL + kSlots,  // + slot
    BAR_S_FULL = BAR_KV_EMPTY + kSlots,   // + tile (A = 0, B = 1)
    BAR_P_FULL = BAR_S_FULL + 2,    // + tile
    BAR_PV_DONE = BAR_P_FULL + 2,   // + tile
    BAR_O_EMPTY = BAR_PV_DONE + 2,  // + tile
    BAR_MMA_DONE = BAR_O_EMPTY + 2,
    BAR_ML_FULL,   // single-tile segments: slot 1's (max, sum) are in shared memory
    BAR_ML_READ,   // single-tile segments: slot 0 has read O_1 and the (max, sum)
    BAR_COUNT
};
constexpr uint32_t kOffMisc = kOffBar + BAR_COUNT * 8;
constexpr uint32_t kOffML = kOffMisc + 128;  // [2][128] floats: slot 1's row max / sum in single-tile segments

// Position q of the K/V load sequence (q = 2j for K(j), 2j + 1 for V(j)).
__device__ __forceinline__ uint32_t ring_slot(uint32_t q) { return q % kSlots; }
__device__ __forceinline__ uint32_t ring_phase(uint32_t q) { return (q / kSlots) & 1; }
constexpr uint32_t kSmemBytes = kOffML + 1024 + 1024;  // + slack to align the base to 1024 bytes

constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t tmem_s(int x) { return (uint32_t)x * 256; }        // S_x, P_x over its first 64
__host__ __device__ constexpr uint32_t tmem_o(int x) { return (uint32_t)x * 256 + 128; }  // O_x

// Shared-memory descriptor halves of the 128-byte-swizzled operand tiles (the fields of
// sdesc_kmajor_sw128 / sdesc_mnmajor_sw128): high half SBO = 1024 bytes, the fixed
// version bit and the swizzle mode; low half leading byte offset (K-major: unused, 1;
// MN-major: the 64-column block stride) above the start address, which is added in.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
constexpr uint32_t kDescLoK = 1u << 16;
constexpr uint32_t kDescLoV = (kHalfBytes >> 4) << 16;
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
    const uint32_t *mask;   // null: ancestor bits from parent
    const int32_t *parent;
    uint16_t *o;
    float *lse;
    int32_t *status;
    uint8_t *ws;  // one block of kWsBlock bytes per CTA (ws_cnt, ws_piece_o, ws_piece_lse)
    int nb, B, Hq, Hkv, G, NT, MT, W, max_pages, num_blocks;
    int unit_aligned;  // 1: group k is exactly unit k (sequence k / Hkv, kv head k % Hkv); nothing is cut
    int merge_in_place;  // 1: the warp whose piece of a cut tile lands last merges it; 0: the merge kernel does
    int kv_evict_first;  // 1: one pair tile per unit, so each K/V page is read once: loaded evict-first in L2
    float scale_log2;
};

// ------------------------------------------------------------------ workspace

// CTA c's block of the workspace: arrival counters, then four piece slots (slot
// 2 * (starts its tile) + x) of normalised O in fp16, chunk-major (8-column chunk k of
// row r at [k][r], so a warp's 32 rows store 512 contiguous bytes per instruction), then
// their LSEs.  A block's counters sit at the same offset whatever the shape or the CTA
// count, so a workspace zeroed once keeps them zero from call to call: every counter
// that is counted up is set back to zero by the warp that merges.
constexpr size_t kWsCntBytes = 128;                           // 8 counters used: [x][quarter]
constexpr size_t kWsSlotO = (size_t)kM * kHeadDim * 2;         // 32 KB
constexpr size_t kWsBlock = kWsCntBytes + 4 * kWsSlotO + 4 * (size_t)kM * sizeof(float);

__device__ __forceinline__ uint32_t *ws_cnt(uint8_t *ws, int cta)
{
    return reinterpret_cast<uint32_t *>(ws + (size_t)cta * kWsBlock);
}
__device__ __forceinline__ uint4 *ws_piece_o(uint8_t *ws, int cta, int slot)
{
    return reinterpret_cast<uint4 *>(ws + (size_t)cta * kWsBlock + kWsCntBytes + (size_t)slot * kWsSlotO);
}
__device__ __forceinline__ float *ws_piece_lse(uint8_t *ws, int cta, int slot)
{
    return reinterpret_cast<float *>(ws + (size_t)cta * kWsBlock + kWsCntBytes + 4 * kWsSlotO) + (size_t)slot * kM;
}

// ------------------------------------------------------------------ schedule

struct Sched {
    const int32_t *prefix_lens;
    int nb, B, Hkv, NT, MT, max_tokens;
    int NP;  // pair tiles per unit: (MT + 1) / 2
};

__device__ __forceinline__ int mtile_tiles(int P, int B, int NT, int mt)
{
    const int kv_end = min(B, (mt + 1) * NT);  // tree keys a node of this M tile can see end here
    return (P + kv_end + kN - 1) / kN;
}

// KV tiles of pair tile mp (its later M tile needs the most keys).
__device__ __forceinline__ int pair_tiles(const Sched &s, int P, int mp)
{
    return mtile_tiles(P, s.B, s.NT, min(2 * mp + 1, s.MT - 1));
}

// Group items of one (sequence, kv head) unit: the KV tiles of its last pair tile, which
// needs the most keys; 0 for a sequence whose prefix does not fit its block table
// (reported as TV_ERR_INVALID_ARG).
__device__ __forceinline__ int unit_tiles(const Sched &s, int P)
{
    if (P < 0 || P > s.max_tokens - s.B) return 0;
    return pair_tiles(s, P, s.NP - 1);
}

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Total group items.  Whole warp.
__device__ long long sched_total(const Sched &s, int lane)
{
    long long tot = 0;
    for (int base = 0; base < s.nb; base += 32) {
        const int b = base + lane;
        const long long t = (b < s.nb) ? (long long)s.Hkv * unit_tiles(s, __ldcg(s.prefix_lens + b)) : 0;
        tot += warp_sum_ll(t);
    }
    return tot;
}

// Sequence and offset inside it of global group item t (t < total).  Whole warp.
__device__ void sched_locate(const Sched &s, long long t, int lane, int &b_out, long long &off_out)
{
    long long acc = 0;
    for (int base = 0; base < s.nb; base += 32) {
        const int b = base + lane;
        const long long tb = (b < s.nb) ? (long long)s.Hkv * unit_tiles(s, __ldcg(s.prefix_lens + b)) : 0;
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

// Groups that get work: at least kMinTilesPerCta group items each, at most `groups`.
__device__ __forceinline__ long long active_groups(long long total, int groups)
{
    long long c = (total + kMinTilesPerCta - 1) / kMinTilesPerCta;
    if (c > groups) c = groups;
    return c < 1 ? 1 : c;
}

// Groups the grid forms: NP CTAs each (one per pair tile of a unit), or a single group
// whose lanes the grid's CTAs share when the grid is smaller than NP.
__device__ __forceinline__ int grid_groups(int grid, int NP) { return grid >= NP ? grid / NP : 1; }

// Group containing group item t, when `total` items are cut evenly into G groups.
__device__ __forceinline__ long long group_of(long long t, long long total, long long G)
{
    return ((t + 1) * G - 1) / total;
}

struct Cursor {
    int b;
    long long off;   // group-item offset inside sequence b
    long long left;  // group items this CTA still has to visit for its current lane
    int lane;        // the pair tile (of every unit) this CTA computes
    int lane_step;   // next lane: lane + lane_step (only when the grid is smaller than NP)
    int b0;          // the range's start and length, to revisit it for the next lane
    long long off0, left0;
    long long sbase, sbase0;  // global index of sequence b's (b0's) first group item
};

struct Seg {
    int b, g, mp, j0, j1, n_row, P;
    bool has_b;
    long long su;  // global index of the unit's first group item
};

// Next segment (a run of KV tiles of one pair tile) of this CTA's share.  A group's CTAs
// walk the same range of group items -- (sequence, kv head, KV tile) ascending -- each for
// its own pair tile of every unit in it, so they read the same K/V pages at about the same
// time and all but the first find them in L2.  A pair tile skips the unit's last tiles when
// only later pair tiles need them.
__device__ __forceinline__ bool next_seg(const Sched &s, Cursor &c, Seg &sg)
{
    for (;;) {
        while (c.left > 0 && c.b < s.nb) {
            const int P = __ldcg(s.prefix_lens + c.b);
            const int ut = unit_tiles(s, P);
            if (c.off >= (long long)ut * s.Hkv) {
                c.sbase += (long long)ut * s.Hkv;
                ++c.b;
                c.off = 0;
                continue;
            }
            const int g = (int)(c.off / ut);
            const int rem = (int)(c.off - (long long)g * ut);
            const int take = (int)min((long long)(ut - rem), c.left);
            c.off += take;
            c.left -= take;
            const int n = pair_tiles(s, P, c.lane);
            if (rem >= n) continue;  // tiles only this unit's later pair tiles need
            sg.b = c.b;
            sg.g = g;
            sg.mp = c.lane;
            sg.j0 = rem;
            sg.j1 = min(rem + take, n);
            sg.n_row = n;
            sg.P = P;
            sg.has_b = 2 * c.lane + 1 < s.MT;
            sg.su = c.sbase + (long long)g * ut;
            return true;
        }
        if (c.left0 <= 0 || c.lane + c.lane_step >= s.NP) return false;
        c.lane += c.lane_step;
        c.b = c.b0;
        c.off = c.off0;
        c.left = c.left0;
        c.sbase = c.sbase0;
    }
}

constexpr int kMaxMaskWords = 8;  // ceil(256 / 32)

// Node i's ancestor bits (i included) from a walk up its root path, into registers
// (word w of the row in m[w]).  Indices must fall strictly along the walk and end at
// the root (parent -1); otherwise the walk stops and TV_ERR_NOT_TOPOLOGICAL is reported.
__device__ __forceinline__ void row_mask_from_parents(const int32_t *__restrict__ par, int i,
                                                      uint32_t (&m)[kMaxMaskWords], int32_t *status)
{
#pragma unroll
    for (int w = 0; w < kMaxMaskWords; ++w) m[w] = 0u;
    for (int j = i;;) {
        const int wj = j >> 5;
        const uint32_t bit = 1u << (j & 31);
#pragma unroll
        for (int w = 0; w < kMaxMaskWords; ++w)
            if (w == wj) m[w] |= bit;
        const int pj = __ldg(par + j);
        if (pj < 0 || pj >= j) {
            if (j != 0 || pj != -1) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
            return;
        }
        j = pj;
    }
}

__device__ __forceinline__ uint32_t word_at(const uint32_t (&m)[kMaxMaskWords], int w)
{
    uint32_t r = 0u;
#pragma unroll
    for (int k = 0; k < kMaxMaskWords; ++k)
        if (k == w) r = m[k];
    return r;
}

// visible_bits (below) with the row's words in registers
__device__ __forceinline__ uint32_t visible_bits_reg(int kstart, int P, int B, const uint32_t (&m)[kMaxMaskWords],
                                                     int W)
{
    if (kstart + 32 <= P) return 0xffffffffu;
    uint32_t v = (kstart >= P) ? 0u : ((1u << (P - kstart)) - 1u);
    const int t0 = kstart - P;
    if (t0 + 32 > 0 && t0 < B) {
        uint32_t bits;
        if (t0 >= 0) {
            const int w = t0 >> 5, sh = t0 & 31;
            const uint32_t lo = word_at(m, w);
            const uint32_t hi = (w + 1 < W) ? word_at(m, w + 1) : 0u;
            bits = sh ? ((lo >> sh) | (hi << (32 - sh))) : lo;
        } else {
            bits = word_at(m, 0) << (-t0);
        }
        v |= bits;
    }
    return v;
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

// ------------------------------------------------------------------ merge

// The split-KV combine of one row of a cut M tile, over the pieces of groups k0 .. k1
// (group k's piece is in CTA k * NP + pm, slot 2 * (k == k0) + x): with lse_k the
// pieces' log-sum-exps and O_k their normalised outputs, lse = ln sum_k e^{lse_k} and
// O = sum_k e^{lse_k - lse} O_k.  One pass per 64 columns over pairs of pieces, each
// pair's LSEs and outputs loaded together, with a running maximum that rescales the
// sums between pairs.  A piece whose keys were all masked has lse_k = -inf and weight
// 0; a row with no visible key at all gets O = 0 and lse = -inf.
__device__ __noinline__ void merge_pieces(uint8_t *ws, int k0, int k1, int NP, int pm, int x, int row,
                                          uint4 *__restrict__ o_row, float *__restrict__ lse_out)
{
    float m = -INFINITY, wsum = 0.f;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        float acc[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) acc[e] = 0.f;
        m = -INFINITY;
        wsum = 0.f;
#pragma unroll 1
        for (int k = k0; k <= k1; k += 2) {
            float l[2];
            uint4 v[2][8];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool in = k + u <= k1;
                const int kk = in ? k + u : k;
                const int cta = kk * NP + pm, slot = (kk == k0 ? 2 : 0) + x;
                l[u] = in ? __ldcg(ws_piece_lse(ws, cta, slot) + row) : -INFINITY;
                const uint4 *src = ws_piece_o(ws, cta, slot) + (size_t)(h * 8) * kM + row;
#pragma unroll
                for (int c = 0; c < 8; ++c) v[u][c] = in ? __ldcg(src + (size_t)c * kM) : make_uint4(0u, 0u, 0u, 0u);
            }
            const float mb = fmaxf(m, fmaxf(l[0], l[1]));
            if (mb == -INFINITY) continue;  // no piece with a visible key yet
            const float sc = expf(m - mb);   // 0 while m is still -inf
            wsum *= sc;
#pragma unroll
            for (int e = 0; e < 64; ++e) acc[e] *= sc;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float w = expf(l[u] - mb);  // 0 for an empty piece
                wsum += w;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float2 a = unpack_f16x2(v[u][c].x), b = unpack_f16x2(v[u][c].y);
                    const float2 d = unpack_f16x2(v[u][c].z), e = unpack_f16x2(v[u][c].w);
                    acc[8 * c + 0] = fmaf(w, a.x, acc[8 * c + 0]);
                    acc[8 * c + 1] = fmaf(w, a.y, acc[8 * c + 1]);
                    acc[8 * c + 2] = fmaf(w, b.x, acc[8 * c + 2]);
                    acc[8 * c + 3] = fmaf(w, b.y, acc[8 * c + 3]);
                    acc[8 * c + 4] = fmaf(w, d.x, acc[8 * c + 4]);
                    acc[8 * c + 5] = fmaf(w, d.y, acc[8 * c + 5]);
                    acc[8 * c + 6] = fmaf(w, e.x, acc[8 * c + 6]);
                    acc[8 * c + 7] = fmaf(w, e.y, acc[8 * c + 7]);
                }
            }
            m = mb;
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 q;
            q.x = pack_bf16x2(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv);
            q.y = pack_bf16x2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
            q.z = pack_bf16x2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
            q.w = pack_bf16x2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
            o_row[h * 8 + c] = q;
        }
    }
    *lse_out = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kThreads, 1) tree_attn_kernel(const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + kOffQ, sKV = base + kOffKV;
    const uint32_t sBar = base + kOffBar;
#define BAR(i) (sBar + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kOffMisc + 4);
    int *sh_b0 = reinterpret_cast<int *>(gbase + kOffMisc + 8);
    long long *sh_off0 = reinterpret_cast<long long *>(gbase + kOffMisc + 16);
    long long *sh_left = reinterpret_cast<long long *>(gbase + kOffMisc + 24);
    int *sh_lane = reinterpret_cast<int *>(gbase + kOffMisc + 32);
    int *sh_step = reinterpret_cast<int *>(gbase + kOffMisc + 36);
    long long *sh_sbase = reinterpret_cast<long long *>(gbase + kOffMisc + 40);
    long long *sh_total = reinterpret_cast<long long *>(gbase + kOffMisc + 48);   // group items
    long long *sh_groups = reinterpret_cast<long long *>(gbase + kOffMisc + 56);  // groups with work

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Sched sch{p.prefix_lens, p.nb, p.B, p.Hkv, p.NT, p.MT, p.max_pages * kPage, (p.MT + 1) / 2};

    if (threadIdx.x == 0) {
        mbar_init(BAR(BAR_Q_FULL), 1);
        mbar_init(BAR(BAR_Q_EMPTY), 1);
        for (int q = 0; q < kSlots; ++q) {
            mbar_init(BAR(BAR_KV_FULL + q), 1);
            mbar_init(BAR(BAR_KV_EMPTY + q), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(BAR(BAR_S_FULL + x), 1);
            mbar_init(BAR(BAR_P_FULL + x), kSoftmaxWarps);
            mbar_init(BAR(BAR_PV_DONE + x), 1);
            mbar_init(BAR(BAR_O_EMPTY + x), kSoftmaxWarps);
        }
        mbar_init(BAR(BAR_MMA_DONE), 1);
        mbar_init(BAR(BAR_ML_FULL), kSoftmaxWarps);
        mbar_init(BAR(BAR_ML_READ), kSoftmaxWarps);
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
    // This kernel is launched as a programmatic dependent of the previous kernel in the
    // stream (normally tv_build_mask), which waits for everything before it and then
    // lets this grid start.  So q, K/V, the block table and prefix_lens (inputs written
    // before that kernel) are read at once (through L2: TMA, __ldcg); only the ancestor
    // masks (or the parent array), which that kernel may still be writing, wait for it
    // (griddepcontrol.wait before the first masked tile, or without a mask array at the
    // start of a segment that reaches the tree keys, and in every thread before it exits).
    if (warp == 2) {
        // CTA c runs lane (pair tile) c % NP of group c / NP; each group takes an equal
        // share of the group items.  A grid smaller than NP forms one group whose lanes
        // its CTAs take in turn.
        // Small launches (p.unit_aligned, chosen by the host) instead give group k exactly
        // unit k, so no tile is cut and no merge is needed.
        const int grid = (int)gridDim.x;
        const int grp = grid >= sch.NP ? (int)blockIdx.x / sch.NP : 0;
        const int lane0 = grid >= sch.NP ? (int)blockIdx.x % sch.NP : (int)blockIdx.x;
        long long t0 = 0, t1 = 0, total = 0, G = 1;
        int b0 = sch.nb;
        long long off0 = 0;
        if (p.unit_aligned) {
            const int bb = grp / sch.Hkv;
            if (bb < sch.nb) {
                const int ut = unit_tiles(sch, __ldcg(sch.prefix_lens + bb));
                if (ut > 0) {
                    b0 = bb;
                    off0 = (long long)(grp % sch.Hkv) * ut;
                    t1 = ut;
                }
            }
        } else {
            total = sched_total(sch, lane);
            G = active_groups(total, grid_groups(grid, sch.NP));
            if (grp < G) {
                t0 = total * grp / G;
                t1 = total * (grp + 1) / G;
            }
            if (t1 > t0) sched_locate(sch, t0, lane, b0, off0);
        }
        if (lane == 0) {
            *sh_b0 = b0;
            *sh_off0 = off0;
            *sh_left = t1 - t0;
            *sh_lane = lane0;
            *sh_step = grid >= sch.NP ? sch.NP : grid;
            *sh_sbase = t0 - off0;  // (stream-K) t0 is item off0 of sequence b0
            *sh_total = total;
            *sh_groups = G;
        }
        if (blockIdx.x == 0) {
            for (int b = lane; b < sch.nb; b += 32) {
                const int P = __ldcg(sch.prefix_lens + b);
                if (P < 0 || P > sch.max_tokens - sch.B) report_status(p.status, TV_ERR_INVALID_ARG);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Cursor cur0{*sh_b0, *sh_off0, *sh_left, *sh_lane, *sh_step, *sh_b0, *sh_off0, *sh_left, *sh_sbase, *sh_sbase};
    pdl_launch_dependents();

    if (warp == 0 || warp == 2) {
        // ---------------------------------------------------------- TMA producers
        // Warp 0 loads Q and the K tiles, warp 2 the V tiles.  A 16-row page half is a
        // 2 KB copy, and one warp issues them at ~26 B/clk/SM on GB300, below the MMA
        // loop's need; two issuing warps overlap their copies.  Each warp waits its own
        // ring positions in order, and positions are released in order (by the MMA warp, or
        // in pair segments by slot 1's softmax), so no wait can alias a later phase of its
        // slot.
        regs_decrease<kRegsLow>();
        const int kvh = warp == 0 ? 0 : 1;
        const uint64_t kv_pol = p.kv_evict_first ? l2_policy_evict_first() : 0ull;
        Cursor cur = cur0;
        Seg sg;
        uint32_t kv = 0, seg_i = 0;
        bool ok = true;
        const int oob_row = p.num_blocks * p.Hkv * kPage;  // first row past the cache: zero fill
        while (ok && next_seg(sch, cur, sg)) {
            if (kvh == 0 && seg_i > 0 && !mbar_wait(BAR(BAR_Q_EMPTY), (seg_i - 1) & 1, abort_flag, p.status)) break;
            if (kvh == 0 && lane == 0) {
                mbar_arrive_expect_tx(BAR(BAR_Q_FULL), kTileBytes * (sg.has_b ? 2 : 1));
                for (int x = 0; x < (sg.has_b ? 2 : 1); ++x) {
                    const int node0 = (2 * sg.mp + x) * p.NT;
                    tma_load_4d(sQ + x * kTileBytes, &p.tm_q, 0, sg.g * p.G, node0, sg.b, BAR(BAR_Q_FULL));
                    tma_load_4d(sQ + x * kTileBytes + kHalfBytes, &p.tm_q, 64, sg.g * p.G, node0, sg.b,
                                BAR(BAR_Q_FULL));
                }
            }
            const int kv_len = sg.P + min(p.B, (2 * sg.mp + (sg.has_b ? 2 : 1)) * p.NT);
            // Physical row of page pg for this kv head, or the zero-filled row past the cache.
            // Lane l holds page (jb * 8 + l) of a 4-tile batch starting at tile jb; the next
            // batch is requested one batch ahead so block-table latency stays off the TMA path.
            auto page_row = [&](int jb) -> int {
                const int pg = jb * (kN / kPage) + lane;
                int r = oob_row;
                if (pg * kPage < kv_len) {
                    const int id = __ldcg(p.block_table + (size_t)sg.b * p.max_pages + pg);
                    if (id >= 0 && id < p.num_blocks)
                        r = (id * p.Hkv + sg.g) * kPage;
                    else
                        report_status(p.status, TV_ERR_INVALID_ARG);
                }
                return r;
            };
            int rows_cur = page_row(sg.j0);
            int rows_nxt = (sg.j0 + 4 < sg.j1) ? page_row(sg.j0 + 4) : oob_row;
            for (int j = sg.j0; j < sg.j1; ++j, ++kv) {
                const int in_batch = (j - sg.j0) & 3;
                if (in_batch == 0 && j != sg.j0) {
                    rows_cur = rows_nxt;
                    rows_nxt = (j + 4 < sg.j1) ? page_row(j + 4) : oob_row;
                }
                const int my_row = __shfl_sync(0xffffffffu, rows_cur, in_batch * 8 + (lane >> 1));
                const uint32_t dst_off = (uint32_t)(lane & 1) * kHalfBytes + (uint32_t)(lane >> 1) * (kPage * 128);
                const uint32_t q = 2 * kv + kvh;  // ring position of K(j) or V(j)
                const uint32_t sl = ring_slot(q);
                if (!mbar_wait(BAR(BAR_KV_EMPTY + sl), ring_phase(q) ^ 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(BAR(BAR_KV_FULL + sl), kTileBytes);
                __syncwarp();
                if (lane < 16) {
                    const void *tm = kvh ? (const void *)&p.tm_v : (const void *)&p.tm_k;
                    const uint32_t dst = sKV + sl * kTileBytes + dst_off;
                    if (p.kv_evict_first)
                        tma_load_2d_hint(dst, tm, (lane & 1) * 64, my_row, BAR(BAR_KV_FULL + sl), kv_pol);
                    else
                        tma_load_2d(dst, tm, (lane & 1) * 64, my_row, BAR(BAR_KV_FULL + sl));
                }
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
        // Slots x = 0, 1 own S_x / O_x.  Pair segments: slot x is M tile x over every
        // KV tile.  Single-tile segments: both slots use Q tile A, slot x takes the KV
        // tiles t with t % 2 == x, and the softmax warpgroups merge at the end.
        // tcgen05.mma issue stalls while the tensor pipe is busy, so everything this warp
        // does between two MMA groups is pipe idle time: a slot's PV(t) and its next QK
        // go out back to back under one commit (S_FULL, which the softmax needs anyway),
        // a step's K/V waits are done once up front, and PV_DONE is committed only after a
        // slot's last PV of the segment.  A commit costs the pipe about as much as an MMA, so
        // in pair segments the ring slots are released by slot 1's softmax instead (S_FULL_1(t)
        // completes only after every MMA before QK_1(t), which includes all readers of V(t-1)
        // and K(t)); single-tile segments release them here, after their readers.
        // The warp shares its SM sub-partition with two softmax warps, so its own
        // instruction count matters too: ring positions advance incrementally and the
        // descriptors come from one register.  The control flow stays warp-uniform (lane 0
        // alone issues), which lets the loop's invariants live in uniform registers.
        regs_decrease<kRegsLow>();
        {
            Cursor cur = cur0;
            Seg sg;
            uint32_t kv = 0, seg_i = 0;
            // tiles and segments per slot so far (barrier phases)
            uint32_t gs0 = 0, gs1 = 0, sc0 = 0, sc1 = 0;
            bool ok = true;
            auto wait_bar = [&](int idx, uint32_t parity) { return mbar_wait(BAR(idx), parity, abort_flag, p.status); };
            // ring position q: K(j) = 2j, V(j) = 2j + 1 (KV tile counter j over the whole CTA)
            struct RingPos {
                uint32_t slot, phase;  // q % kSlots, (q / kSlots) & 1
            };
            auto at = [](uint32_t q) { return RingPos{q % kSlots, (q / kSlots) & 1u}; };
            auto ahead = [](RingPos r, uint32_t d) {  // position q + d, d < kSlots
                r.slot += d;
                if (r.slot >= (uint32_t)kSlots) {
                    r.slot -= kSlots;
                    r.phase ^= 1u;
                }
                return r;
            };
            auto full = [&](RingPos r) { return wait_bar(BAR_KV_FULL + r.slot, r.phase); };
            // Descriptors: the high halves are constants and every low half is the
            // 1024-aligned shared-memory base (in 16-byte units) plus a constant, so one
            // register holds them all (this warp runs in 64 registers); only the
            // start-address field moves per K slice (see umma_bf16_ss_lohi).
            const uint32_t d0 = base >> 4;
            auto qk = [&](int x, int qx, RingPos rk) {  // S_x = Q_qx K^T, K in ring slot rk
                const uint32_t qa = d0 + kDescLoK + ((kOffQ + qx * kTileBytes) >> 4);
                const uint32_t ka = d0 + kDescLoK + (kOffKV >> 4) + rk.slot * (kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    umma_bf16_ss_lohi(tmem + tmem_s(x), qa + off, kDescHi, ka + off, kDescHi, kIdescQK,
                                      kk > 0 ? 1u : 0u);
                }
            };
            auto pv = [&](int x, RingPos rv, bool accumulate) {  // O_x (+)= P_x V, V in ring slot rv
                const uint32_t va = d0 + kDescLoV + (kOffKV >> 4) + rv.slot * (kTileBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk)
                    umma_bf16_ts_lohi(tmem + tmem_o(x), tmem + tmem_s(x) + kk * 8, va + kk * (2048 >> 4), kDescHi,
                                      kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
            };
            while (ok && next_seg(sch, cur, sg)) {
                const int n = sg.j1 - sg.j0;
                const bool pair = sg.has_b;
                const int nx0 = pair ? n : (n + 1) / 2, nx1 = pair ? n : n / 2;
                if (!wait_bar(BAR_Q_FULL, seg_i & 1)) { ok = false; break; }
                const RingPos r0 = at(2 * kv);  // K of the segment's first tile
                if (pair) {
                    if (!full(r0)) { ok = false; break; }
                    tc_fence_after();
                    if (lane == 0) {
                        qk(0, 0, r0);
                        umma_commit(BAR(BAR_S_FULL + 0));
                        qk(1, 1, r0);
                        umma_commit(BAR(BAR_S_FULL + 1));
                        if (n == 1) umma_commit(BAR(BAR_Q_EMPTY));
                    }
                    __syncwarp();
                    // Per step t the waits before a group go out as one try_wait over the
                    // warp's lanes (each lane names its own barrier).
                    RingPos rv = ahead(r0, 1), rk = ahead(r0, 2);  // V(t), K(t + 1)
                    for (int t = 0; t < n; ++t) {
                        const bool more = t + 1 < n;
                        // lane 0: V(t); lane 1: K(t + 1); lane 2: slot 0's P(t); lane 3: slot 0's O
                        // read by the previous segment's epilogue (first tile only)
                        uint32_t wb = BAR(BAR_KV_FULL + rv.slot), wp = rv.phase;
                        if (lane == 1 && more) {
                            wb = BAR(BAR_KV_FULL + rk.slot);
                            wp = rk.phase;
                        } else if (lane == 2) {
                            wb = BAR(BAR_P_FULL + 0);
                            wp = (gs0 + t) & 1;
                        } else if (lane == 3 && t == 0 && sc0 > 0) {
                            wb = BAR(BAR_O_EMPTY + 0);
                            wp = (sc0 - 1) & 1;
                        }
                        if (!mbar_wait_lanes(wb, wp, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        if (lane == 0) {
                            pv(0, rv, t > 0);
                            if (more) {
                                qk(0, 0, rk);
                                umma_commit(BAR(BAR_S_FULL + 0));
                            } else {
                                umma_commit(BAR(BAR_PV_DONE + 0));
                            }
                        }
                        __syncwarp();
                        // lane 0: slot 1's P(t); lane 1: slot 1's O (first tile only)
                        wb = BAR(BAR_P_FULL + 1);
                        wp = (gs1 + t) & 1;
                        if (lane == 1 && t == 0 && sc1 > 0) {
                            wb = BAR(BAR_O_EMPTY + 1);
                            wp = (sc1 - 1) & 1;
                        }
                        if (!mbar_wait_lanes(wb, wp, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        if (lane == 0) {
                            pv(1, rv, t > 0);
                            if (more) {
                                qk(1, 1, rk);
                                umma_commit(BAR(BAR_S_FULL + 1));
                            } else {
                                umma_commit(BAR(BAR_PV_DONE + 1));
                            }
                            if (t + 2 == n) umma_commit(BAR(BAR_Q_EMPTY));
                        }
                        __syncwarp();
                        rv = ahead(rv, 2);
                        rk = ahead(rk, 2);
                    }
                } else {
                    // issue order: QK_0(0), QK_1(1), then per tile t: PV_{t%2}(t), QK_{t%2}(t+2)
                    const RingPos r2 = ahead(r0, 2);  // K of the second tile
                    if (!full(r0) || (n > 1 && !full(r2))) { ok = false; break; }
                    tc_fence_after();
                    if (lane == 0) {
                        qk(0, 0, r0);
                        umma_commit(BAR(BAR_S_FULL + 0));
                        umma_commit(BAR(BAR_KV_EMPTY + r0.slot));
                        if (n > 1) {
                            qk(1, 0, r2);
                            umma_commit(BAR(BAR_S_FULL + 1));
                            umma_commit(BAR(BAR_KV_EMPTY + r2.slot));
                        }
                        if (n <= 2) umma_commit(BAR(BAR_Q_EMPTY));
                    }
                    __syncwarp();
                    RingPos rv = ahead(r0, 1), rk = ahead(r0, 4);  // V(t), K(t + 2)
                    for (int t = 0; t < n; ++t) {
                        const int x = t & 1;
                        const bool more = t + 2 < n;
                        // PV(t) waits only for V(t): these segments are bandwidth-bound, and K(t+2)
                        // is two tiles further out in the ring
                        // lane 0: V(t); lane 1: slot x's P; lane 2: slot x's O read by the previous
                        // segment's epilogue (the slot's first tile only)
                        {
                            const int lx = t >> 1;
                            const uint32_t gsx = x ? gs1 : gs0, scx = x ? sc1 : sc0;
                            uint32_t wb = BAR(BAR_KV_FULL + rv.slot), wp = rv.phase;
                            if (lane == 1) {
                                wb = BAR(BAR_P_FULL + x);
                                wp = (gsx + lx) & 1;
                            } else if (lane == 2 && lx == 0 && scx > 0) {
                                wb = BAR(BAR_O_EMPTY + x);
                                wp = (scx - 1) & 1;
                            }
                            if (!mbar_wait_lanes(wb, wp, abort_flag, p.status)) { ok = false; break; }
                        }
                        tc_fence_after();
                        if (lane == 0) {
                            pv(x, rv, t > 1);
                            if (!more) umma_commit(BAR(BAR_PV_DONE + x));
                            umma_commit(BAR(BAR_KV_EMPTY + rv.slot));
                        }
                        __syncwarp();
                        if (more) {
                            if (!full(rk)) { ok = false; break; }
                            tc_fence_after();
                            if (lane == 0) {
                                qk(x, 0, rk);
                                umma_commit(BAR(BAR_S_FULL + x));
                                umma_commit(BAR(BAR_KV_EMPTY + rk.slot));
                                if (t + 3 == n) umma_commit(BAR(BAR_Q_EMPTY));
                            }
                            __syncwarp();
                        }
                        rv = ahead(rv, 2);
                        rk = ahead(rk, 2);
                    }
                }
                if (!ok) break;
                kv += n;
                gs0 += nx0;
                gs1 += nx1;
                if (nx0 > 0) ++sc0;
                if (nx1 > 0) ++sc1;
                ++seg_i;
            }
            // Every MMA this CTA issued completes before TMEM is released.
            if (lane == 0) umma_commit(BAR(BAR_MMA_DONE));
            __syncwarp();
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(BAR(BAR_MMA_DONE), 0) && global_timer_ns() - t0 < kWaitLimitNs) { }
        }
    } else if (warp == 3) {
        regs_decrease<kRegsLow>();
    } else {
        // ------------------------------------------------ softmax + epilogue of slot x
        regs_increase<kRegsHigh>();
        const int x = (warp - 4) >> 2;
        const int row = threadIdx.x - 128 * (1 + x);
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t col_s = tmem_s(x), col_o = tmem_o(x);
        const int node_local = row / p.G;
        const int hg = row - node_local * p.G;
        const float sl2 = p.scale_log2;
        const long long s_total = *sh_total, s_groups = *sh_groups;
        float *sh_m = reinterpret_cast<float *>(gbase + kOffML);  // slot 1's running max / sum per row
        float *sh_l = sh_m + kM;
        Cursor cur = cur0;
        Seg sg;
        // gx: this slot's tiles so far; sx: segments with tiles for this slot; n_merge:
        // single-tile hand-overs so far (ML_* phases)
        uint32_t gx = 0, sx = 0, n_merge = 0;
        uint32_t kvs = 0;  // KV tiles of the CTA's earlier segments (ring positions 2 kvs on)
        // Pair segments: this thread (slot 1, row 0) releases the ring slots of K(t) and V(t-1)
        // once S_1(t) is complete, and the last V once the slot's last PV is.
        const bool releaser = x == 1 && row == 0;
        auto release = [&](uint32_t q) { mbar_arrive(BAR(BAR_KV_EMPTY + ring_slot(q))); };
        // primary_done: this thread has waited for the previous kernel (griddepcontrol.wait),
        // before its first read of the masks or parents and before its first global write
        bool ok = true, primary_done = false;
        while (ok && next_seg(sch, cur, sg)) {
            const int n = sg.j1 - sg.j0;
            const bool pair = sg.has_b;
            const int nx = pair ? n : (x == 0 ? (n + 1) / 2 : n / 2);
            if (nx == 0) {  // slot unused in this segment
                kvs += n;
                continue;
            }
            const int i = (2 * sg.mp + (pair ? x : 0)) * p.NT + node_local;
            const bool valid = i < p.B;
            const uint32_t *mrow = p.mask ? p.mask + ((size_t)sg.b * p.B + (valid ? i : 0)) * p.W : nullptr;
            uint32_t mreg[kMaxMaskWords];  // the row's ancestor bits when there is no mask array
            bool mreg_built = false;
            // Without a mask array, a segment that reaches the tree keys walks the row's root
            // path (dependent loads over the parent array) now, while the first S of the
            // segment is still on its way, rather than at its first masked tile.
            if (!mrow && valid && (long long)sg.j1 * kN > sg.P) {
                if (!primary_done) {  // the parents may come from the previous kernel
                    pdl_wait_primary();
                    primary_done = true;
                }
                row_mask_from_parents(p.parent + (size_t)sg.b * p.B, i, mreg, p.status);
                mreg_built = true;
            }
            float m_run = -INFINITY, l_run = 0.f;  // m_run in log2 units of the scaled score
            for (int lx = 0; lx < nx; ++lx) {
                const int t = pair ? lx : 2 * lx + x;
                const uint32_t g_t = gx + lx;
                const int k0 = (sg.j0 + t) * kN;
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(BAR_S_FULL + x), g_t & 1, abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                if (pair && releaser) {
                    if (t > 0) release(2 * (kvs + t) - 1);  // V(t - 1)
                    release(2 * (kvs + t));                 // K(t)
                }
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + col_s + c * 32, s[c]);
                tmem_ld_wait(s[0]);
                reg_order(s[1]);
                reg_order(s[2]);
                reg_order(s[3]);

                // tree / tail mask (prefix-only tiles skip it), then the row max of the raw scores
                if (!(valid && k0 + kN <= sg.P)) {
                    if (!primary_done) {  // the masks (or parents) may come from the previous kernel
                        pdl_wait_primary();
                        primary_done = true;
                    }
                    if (!mrow && valid && !mreg_built) {
                        row_mask_from_parents(p.parent + (size_t)sg.b * p.B, i, mreg, p.status);
                        mreg_built = true;
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t vis = !valid ? 0u
                                             : mrow ? visible_bits(k0 + 32 * c, sg.P, p.B, mrow, p.W)
                                                    : visible_bits_reg(k0 + 32 * c, sg.P, p.B, mreg, p.W);
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c][e] = ((vis >> e) & 1u) ? s[c][e] : 0xff800000u;
                    }
                }
                float mx[4];  // four independent chains of 3-input maxima
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    mx[c] = fmax3(__uint_as_float(s[c][0]), __uint_as_float(s[c][1]), __uint_as_float(s[c][2]));
#pragma unroll
                    for (int e = 3; e < 31; e += 2)
                        mx[c] = fmax3(mx[c], __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
                    mx[c] = fmaxf(mx[c], __uint_as_float(s[c][31]));
                }
                const float tmax = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;

                // move the running max only when it grows by more than 2^8; the commit
                // behind S(t) also covered this slot's previous PV, so O_x is stable here
                const float m_new = fmaxf(m_run, tmax);
                const bool rescale = m_new > m_run + kRescaleLog2;
                float alpha = 1.f;
                if (rescale) {
                    alpha = ex2_approx(m_run - m_new);
                    l_run *= alpha;
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;

                // P = exp2(s * scale * log2 e - m) as bf16 pairs, packed in place (pair e of
                // block c lands in s[c][e], e < 16) and stored over the first 64 columns of S.
                // The scale and the row sum use packed f32x2 math: these warps share each SM
                // sub-partition with the MMA and TMA warps, and every issue slot they leave free
                // lets those keep the tensor pipe and the K/V ring fed.
                const float2 scale2 = make_float2(sl2, sl2), negm2 = make_float2(neg_m, neg_m);
                float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        float2 v = make_float2(__uint_as_float(s[c][2 * e2]), __uint_as_float(s[c][2 * e2 + 1]));
                        v = __ffma2_rn(v, scale2, negm2);
                        v.x = ex2_approx(v.x);
                        v.y = ex2_approx(v.y);
                        if (e2 & 1)
                            lb = __fadd2_rn(lb, v);
                        else
                            la = __fadd2_rn(la, v);
                        s[c][e2] = pack_bf16x2(v.x, v.y);
                    }
                    if (c & 1) tmem_st16x2(lane_addr + col_s + (c >> 1) * 32, s[c - 1], s[c]);
                }
                l_run += (la.x + la.y) + (lb.x + lb.y);
                // O_x *= alpha before PV(t) adds this tile (PV(t) waits for P_FULL below).  TMEM
                // loads/stores are warp-wide (.sync.aligned), so the whole warp takes the branch
                // when any lane needs it, each lane with its own factor.  Before this slot's first
                // PV of the segment O_x holds nothing (that PV overwrites it).
                if (lx > 0 && __any_sync(0xffffffffu, rescale && alpha < 1.f)) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(lane_addr + col_o + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(lane_addr + col_o + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(BAR_P_FULL + x));
            }
            if (!ok) break;

            // epilogue: O_x of this segment is complete once its last PV lands (one PV_DONE
            // phase per segment in which the slot has tiles)
            if (!__all_sync(0xffffffffu, mbar_wait(BAR(BAR_PV_DONE + x), sx & 1, abort_flag, p.status))) break;
            ++sx;
            if (pair && releaser) release(2 * (kvs + n) - 1);  // V(n - 1)
            const bool merge_slots = !pair && n > 1;  // slot 1 holds the odd KV tiles of the same rows
            if (merge_slots && x == 1) {
                // hand the row's (max, sum) to slot 0, which reads O_1 from TMEM itself
                sh_m[row] = m_run;
                sh_l[row] = l_run;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(BAR_ML_FULL));
                if (!__all_sync(0xffffffffu, mbar_wait(BAR(BAR_ML_READ), n_merge & 1, abort_flag, p.status))) break;
                tc_fence_after();
                if (lane == 0) mbar_arrive(BAR(BAR_O_EMPTY + 1));
                gx += nx;
                kvs += n;
                ++n_merge;
                continue;
            }
            if (merge_slots &&
                !__all_sync(0xffffffffu, mbar_wait(BAR(BAR_ML_FULL), n_merge & 1, abort_flag, p.status)))
                break;
            tc_fence_after();
            // O = (O_0 a0 + O_1 a1) / (l_0 a0 + l_1 a1) when slot 1 holds the odd KV tiles of the
            // same rows (a0, a1 move both halves to the larger max); else O = O_x / l
            float a0 = 1.f, a1 = 0.f;
            if (merge_slots) {
                const float m1 = sh_m[row], l1 = sh_l[row];
                const float mm = fmaxf(m_run, m1);
                a0 = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mm);
                a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - mm);
                l_run = l_run * a0 + l1 * a1;
                m_run = (mm == -INFINITY) ? m_run : mm;
            }
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const float lse_nat = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            const float w0 = a0 * inv, w1 = a1 * inv;
            const int h = sg.g * p.G + hg;
            const size_t orow = ((size_t)sg.b * p.B + i) * p.Hq + h;
            const bool whole = sg.j0 == 0 && sg.j1 == sg.n_row;  // else a piece cut between CTAs
            // A piece is parked in fp16 (it is normalised, |O| <= max|V|).  A CTA's only piece
            // that continues a tile is its first segment and its only piece that starts one
            // is its last, so the slot (2 * starts + x) is unique in the CTA and its owner is
            // known to every other piece of the tile.
            const int wslot = (sg.j0 == 0 ? 2 : 0) + x;
            uint4 *dst_o = reinterpret_cast<uint4 *>(p.o + orow * kHeadDim);
            uint4 *dst_w = ws_piece_o(p.ws, (int)blockIdx.x, wslot) + row;
            if (!primary_done) {  // a kernel before this one may still read what is written here
                pdl_wait_primary();
                primary_done = true;
            }
            // 32 columns at a time: TMEM -> registers -> global
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_addr + col_o + c * 32, o);
                tmem_ld_wait(o);
                if (merge_slots) {
                    uint32_t o1[32];
                    tmem_ld32(lane_addr + tmem_o(1) + c * 32, o1);
                    tmem_ld_wait(o1);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(fmaf(__uint_as_float(o[e]), w0, __uint_as_float(o1[e]) * w1));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * w0);
                }
                if (!valid) continue;
                if (whole) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[q * 8 + 0]), __uint_as_float(o[q * 8 + 1]));
                        v.y = pack_bf16x2(__uint_as_float(o[q * 8 + 2]), __uint_as_float(o[q * 8 + 3]));
                        v.z = pack_bf16x2(__uint_as_float(o[q * 8 + 4]), __uint_as_float(o[q * 8 + 5]));
                        v.w = pack_bf16x2(__uint_as_float(o[q * 8 + 6]), __uint_as_float(o[q * 8 + 7]));
                        dst_o[c * 4 + q] = v;
                    }
                } else {
                    // evict-last: a tile's first pieces wait here while the K/V stream passes
                    // through L2, until the merge reads them
                    const uint64_t pol = l2_policy_evict_last();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 v;
                        v.x = pack_f16x2(__uint_as_float(o[q * 8 + 0]), __uint_as_float(o[q * 8 + 1]));
                        v.y = pack_f16x2(__uint_as_float(o[q * 8 + 2]), __uint_as_float(o[q * 8 + 3]));
                        v.z = pack_f16x2(__uint_as_float(o[q * 8 + 4]), __uint_as_float(o[q * 8 + 5]));
                        v.w = pack_f16x2(__uint_as_float(o[q * 8 + 6]), __uint_as_float(o[q * 8 + 7]));
                        st_global_v4_hint(dst_w + (size_t)(c * 4 + q) * kM, v, pol);
                    }
                }
            }
            if (merge_slots) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(BAR_ML_READ));
                ++n_merge;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(BAR_O_EMPTY + x));
            if (valid) {
                if (whole)
                    p.lse[orow] = lse_nat;
                else
                    ws_piece_lse(p.ws, (int)blockIdx.x, wslot)[row] = lse_nat;
            }
            if (!whole && p.merge_in_place) {
                // The tile's pieces come from groups k0 .. k1 (lane sg.mp of each); this warp's
                // 32 rows count in at group k0's CTA, and the warp that lands last merges them.
                const long long k0 = group_of(sg.su, s_total, s_groups);
                const long long k1 = group_of(sg.su + sg.n_row - 1, s_total, s_groups);
                uint32_t *cnt = ws_cnt(p.ws, (int)k0 * sch.NP + sg.mp) + x * 4 + (warp & 3);
                fence_acq_rel_gpu();  // this warp's piece is visible before it is counted
                __syncwarp();
                uint32_t seen = 0;
                if (lane == 0) seen = atomicAdd(cnt, 1u);
                seen = __shfl_sync(0xffffffffu, seen, 0);
                if (seen == (uint32_t)(k1 - k0)) {
                    fence_acq_rel_gpu();  // every other piece counted in before: read them now
                    if (valid)
                        merge_pieces(p.ws, (int)k0, (int)k1, sch.NP, sg.mp, x, row,
                                     reinterpret_cast<uint4 *>(p.o + orow * kHeadDim), p.lse + orow);
                    if (lane == 0) *cnt = 0u;  // zero again for the next call
                }
            }
            gx += nx;
            kvs += n;
        }
    }

    // no thread exits before the previous kernel has completed, so kernels after this
    // one (which wait only for it) also see that kernel's results
    pdl_wait_primary();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
#undef BAR
}

// ------------------------------------------------------------------ merge kernel

constexpr int kMergeThreads = 128;  // 32 rows x 4 column quarters
constexpr int kMergeSplit = kM / 32; // CTAs per M tile

// Group items before sequence b_end.  Whole warp.
__device__ long long sched_prefix(const Sched &s, int b_end, int lane)
{
    long long tot = 0;
    for (int base = 0; base < b_end; base += 32) {
        const int b = base + lane;
        const long long t = (b < b_end) ? (long long)s.Hkv * unit_tiles(s, __ldcg(s.prefix_lens + b)) : 0;
        tot += warp_sum_ll(t);
    }
    return tot;
}

struct MergeParams {
    const int32_t *prefix_lens;
    uint8_t *ws;
    uint16_t *o;
    float *lse;
    int nb, B, Hq, Hkv, G, NT, MT, max_pages, attn_grid;
};

// The merge of launches whose cut M tiles have many pieces (the attention kernel merges
// in place when they have few: there one warp per 32 rows is fast enough).  kMergeSplit
// CTAs per M tile (sequence, kv head, mt), each for 32 of its rows; thread (warp q, lane
// l) owns row 32s + l and the columns 32q .. 32q+31.  The pieces of a tile whose pair
// tile (lane pm of its unit) was cut come from groups k0 .. k1, group k's in CTA
// k * NP + pm, slot 2 * (k == k0) + x.  The same combine as merge_pieces, in one pass
// over batches of four pieces whose lse and O loads are all in flight together
// (chunk-major partials: a warp's loads are 512 contiguous bytes).
__global__ void __launch_bounds__(kMergeThreads) tree_attn_merge_kernel(const MergeParams mp)
{
    __shared__ int s_k0, s_k1;
    const int id = blockIdx.x / kMergeSplit;
    const int split = blockIdx.x % kMergeSplit;
    const int b = id / (mp.Hkv * mp.MT);
    const int g = (id / mp.MT) % mp.Hkv;
    const int mt = id % mp.MT;
    const int x = mt & 1;
    const int pm = mt >> 1;
    const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
    const Sched sch{mp.prefix_lens, mp.nb, mp.B, mp.Hkv, mp.NT, mp.MT, mp.max_pages * kPage, (mp.MT + 1) / 2};

    pdl_launch_dependents();  // the next kernel (its own wait keeps it ordered) may start launching
    if (q == 0) {  // prefix_lens is an input of both kernels: safe to read before the dependency wait
        const long long total = sched_total(sch, lane);
        const long long G = active_groups(total, grid_groups(mp.attn_grid, sch.NP));
        const long long start_b = sched_prefix(sch, b, lane);
        const int P = __ldcg(mp.prefix_lens + b);
        const int ut = unit_tiles(sch, P);
        int k0 = 0, k1 = 0;
        if (ut > 0 && total > 0) {
            const long long su = start_b + (long long)g * ut;  // the unit's first group item
            k0 = (int)group_of(su, total, G);
            k1 = (int)group_of(su + pair_tiles(sch, P, pm) - 1, total, G);
        }
        if (lane == 0) {
            s_k0 = k0;
            s_k1 = k1;
        }
    }
    __syncthreads();
    const int k0 = s_k0, k1 = s_k1;
    // Every CTA waits for the attention grid (so this grid never completes before it);
    // past this point the partials are complete and visible.
    pdl_wait_primary();
    if (k0 == k1) return;  // the attention kernel wrote this M tile itself
    const int r = split * 32 + lane;
    const int i = mt * mp.NT + r / mp.G;
    if (i >= mp.B) return;  // a row past the tree

    float m = -INFINITY, wsum = 0.f;
    float4 acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int kb = k0; kb <= k1; kb += 4) {
        float l[4];
        uint4 v[4][4];  // 8 fp16 columns each: this thread's 32 columns of 4 pieces
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = kb + u;
            const bool in = k <= k1;
            const int kk = in ? k : k0;
            const int cta = kk * sch.NP + pm, slot = (kk == k0 ? 2 : 0) + x;
            l[u] = in ? __ldcg(ws_piece_lse(mp.ws, cta, slot) + r) : -INFINITY;
            const uint4 *src = ws_piece_o(mp.ws, cta, slot) + (size_t)(q * 4) * kM + r;
#pragma unroll
            for (int c = 0; c < 4; ++c) v[u][c] = in ? __ldcg(src + (size_t)c * kM) : make_uint4(0u, 0u, 0u, 0u);
        }
        const float mb = fmaxf(fmaxf(m, fmaxf(l[0], l[1])), fmaxf(l[2], l[3]));
        if (mb == -INFINITY) continue;  // no piece with a visible key yet
        const float sc = expf(m - mb);  // 0 while m is still -inf
        wsum *= sc;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            acc[k].x *= sc;
            acc[k].y *= sc;
            acc[k].z *= sc;
            acc[k].w *= sc;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float w = expf(l[u] - mb);  // 0 for an empty piece
            wsum += w;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 a = unpack_f16x2(v[u][c].x), bb = unpack_f16x2(v[u][c].y);
                const float2 d = unpack_f16x2(v[u][c].z), e = unpack_f16x2(v[u][c].w);
                acc[2 * c].x = fmaf(w, a.x, acc[2 * c].x);
                acc[2 * c].y = fmaf(w, a.y, acc[2 * c].y);
                acc[2 * c].z = fmaf(w, bb.x, acc[2 * c].z);
                acc[2 * c].w = fmaf(w, bb.y, acc[2 * c].w);
                acc[2 * c + 1].x = fmaf(w, d.x, acc[2 * c + 1].x);
                acc[2 * c + 1].y = fmaf(w, d.y, acc[2 * c + 1].y);
                acc[2 * c + 1].z = fmaf(w, e.x, acc[2 * c + 1].z);
                acc[2 * c + 1].w = fmaf(w, e.y, acc[2 * c + 1].w);
            }
        }
        m = mb;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const size_t orow = ((size_t)b * mp.B + i) * mp.Hq + g * mp.G + r % mp.G;
    uint4 *dst = reinterpret_cast<uint4 *>(mp.o + orow * kHeadDim) + q * 4;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 w4;
        w4.x = pack_bf16x2(acc[2 * c].x * inv, acc[2 * c].y * inv);
        w4.y = pack_bf16x2(acc[2 * c].z * inv, acc[2 * c].w * inv);
        w4.z = pack_bf16x2(acc[2 * c + 1].x * inv, acc[2 * c + 1].y * inv);
        w4.w = pack_bf16x2(acc[2 * c + 1].z * inv, acc[2 * c + 1].w * inv);
        dst[c] = w4;
    }
    if (q == 0) mp.lse[orow] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
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
    (void)row_tiles;
    return (size_t)ctas * kWsBlock;  // per CTA: counters, four fp16 O pieces and their LSEs
}

int attn_row_tiles(const tv_attn_args *a)
{
    const int NT = kM / (a->Hq / a->Hkv);
    return a->nb * a->Hkv * ((a->B + NT - 1) / NT);
}

struct AttnPlan {
    int grid, unit_aligned, merge_in_place, kv_evict_first;
};

// How a call with `ctas` CTAs runs.  A launch whose units all fit the grid at once and
// whose block table covers only a few KV tiles per unit (its length bounds every unit's)
// gives each unit its own CTA group: no tile is cut, so nothing is merged.  Otherwise,
// with G groups over U units a cut tile has about G / U + 1 pieces.  Under three, the
// last piece's warp merges its 32 rows at once (measured faster: no second kernel); from
// three on, that one warp's dependent loads at the grid's tail take longer than the merge
// kernel, which spreads each tile over four CTAs of four warps.  With one pair tile per
// unit every K/V page is read by one CTA only, a stream through L2: those loads are made
// evict-first (measured: the batch-8 and batch-32 workloads' attention 7-9% faster);
// with several, a group's CTAs share each page through L2, and the loads stay normal.
static AttnPlan attn_plan(const tv_attn_args *a, int ctas)
{
    const int NT = kM / (a->Hq / a->Hkv);
    const int MT = (a->B + NT - 1) / NT;
    const int NP = (MT + 1) / 2;
    const long long units = (long long)a->nb * a->Hkv;
    const long long unit_ctas = units * NP;
    const long long max_unit_tiles = ((long long)a->max_pages * kPage + kN - 1) / kN;
    AttnPlan pl;
    pl.unit_aligned = (unit_ctas <= ctas && max_unit_tiles <= kAlignedMaxTiles) ? 1 : 0;
    pl.grid = pl.unit_aligned ? (int)unit_ctas : ctas;
    const long long groups = ctas >= NP ? ctas / NP : 1;
    pl.merge_in_place = (pl.unit_aligned || groups < 2 * units) ? 1 : 0;
    pl.kv_evict_first = NP == 1 ? 1 : 0;
    return pl;
}

int attn_kernel_launches(const tv_attn_args *a, int ctas) { return attn_plan(a, ctas).merge_in_place ? 1 : 2; }

// The attention kernel's shared-memory opt-in, once per device.
static cudaError_t attn_smem_opt_in()
{
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit && (done_mask.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess && bit) done_mask.fetch_or(bit, std::memory_order_relaxed);
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
    p.parent = a->parent_d;
    p.o = static_cast<uint16_t *>(a->o_d);
    p.lse = a->lse_d;
    p.status = a->dev_status_d;
    p.ws = static_cast<uint8_t *>(workspace);
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
    const AttnPlan plan = attn_plan(a, ctas);
    p.unit_aligned = plan.unit_aligned;
    p.merge_in_place = plan.merge_in_place;
    p.kv_evict_first = plan.kv_evict_first;

    cudaError_t e = attn_smem_opt_in();
    if (e == cudaSuccess)
        e = launch_dependent(tree_attn_kernel, dim3(plan.grid), dim3(kThreads), kSmemBytes, stream, p);
    if (e == cudaSuccess && !p.merge_in_place) {
        // The merge kernel may be scheduled while the attention grid drains; it waits
        // (griddepcontrol.wait) before reading partials.
        MergeParams mp{a->prefix_lens_d, p.ws, p.o, p.lse, p.nb, p.B, p.Hq, p.Hkv, p.G, p.NT, p.MT, p.max_pages, ctas};
        e = launch_dependent(tree_attn_merge_kernel, dim3((unsigned)(a->nb * a->Hkv * p.MT * kMergeSplit)),
                             dim3(kMergeThreads), 0, stream, mp);
    }
    if (e != cudaSuccess) {
        *cuda_err = e;
        return TV_ERR_CUDA;
    }
    return TV_OK;
}

}  // namespace tv
