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
//   u_i = beta_i (v_i - gamma_i S0^T k_i - sum_{j strict ancestor} r_ij (k_i . k_j) u_j)
//   o_i = gamma_i S0^T q_i + sum_{j in path(i)} r_ij (q_i . k_j) u_j.
// (X_ij = beta_i r_ij k_i.k_j and Y_ij = r_ij q_i.k_j are the pages' interaction
// matrices, restricted to ancestors by the tree mask.)
//
// GPU form, two kernels on the caller's stream:
//   1. gdn_state_products_kernel: the dense part, K S0 and Q S0 (B x D x D each),
//      one CTA per 32 tree rows of a (sequence, head): S0 staged in shared memory,
//      a 4 x 4 register tile per thread, fp32 into the workspace.
//   2. gdn_tree_solve_kernel: the sparse part, one CTA per (sequence, head), one
//      warp per node in dataflow order: node i waits (bounded) for its parent's
//      done flag, walks up its ancestors forming k_i.k_j and q_i.k_j with warp
//      reductions and the decay ratio r_ij as a running product of alphas (no
//      division), keeps u_i in shared memory for its descendants and writes o_i.
//      Warps take nodes in index order, so the smallest unfinished node can always
//      run: the wait always ends.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kGdnD = 128;
constexpr int kGdnMaxB = 256;
constexpr int kGdnRows = 32;      // tree rows per CTA in the dense kernel
constexpr int kGdnThreads = 256;  // both kernels

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// KS0[i][c] = sum_r k_i[r] S0[r][c], QS0 likewise, for kGdnRows rows of one (b, h).
__global__ void __launch_bounds__(kGdnThreads) gdn_state_products_kernel(const uint16_t *__restrict__ q,
                                                                         const uint16_t *__restrict__ k,
                                                                         const float *__restrict__ S0, int B, int H,
                                                                         float *__restrict__ ks0,
                                                                         float *__restrict__ qs0)
{
    extern __shared__ float4 gdn_smem[];
    float *s_S = reinterpret_cast<float *>(gdn_smem);   // [D][D]
    float *s_kq = s_S + kGdnD * kGdnD;                  // [2][kGdnRows][D] (k rows, then q rows)
    const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int row0 = blk * kGdnRows;
    pdl_wait_primary();
    pdl_launch_dependents();
    const float4 *src = reinterpret_cast<const float4 *>(S0 + ((size_t)b * H + h) * kGdnD * kGdnD);
    for (int t = tid; t < kGdnD * kGdnD / 4; t += kGdnThreads) reinterpret_cast<float4 *>(s_S)[t] = src[t];
    for (int t = tid; t < 2 * kGdnRows * kGdnD; t += kGdnThreads) {
        const int which = t / (kGdnRows * kGdnD), rem = t - which * kGdnRows * kGdnD;
        const int r = rem / kGdnD, d = rem - r * kGdnD;
        const int i = row0 + r;
        float x = 0.f;
        if (i < B) x = bf16_to_f32((which ? q : k)[(((size_t)b * B + i) * H + h) * kGdnD + d]);
        s_kq[t] = x;
    }
    __syncthreads();
    // thread: columns 4*(tid % 32) .. +3, rows 4*(tid / 32) .. +3 of both products
    const int c0 = 4 * (tid & 31), r0 = 4 * (tid >> 5);
    float acc[2][4][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[m][a][c] = 0.f;
#pragma unroll 4
    for (int r = 0; r < kGdnD; ++r) {
        const float4 s = reinterpret_cast<const float4 *>(s_S + r * kGdnD)[c0 / 4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float x = s_kq[(m * kGdnRows + r0 + a) * kGdnD + r];
                acc[m][a][0] = fmaf(x, s.x, acc[m][a][0]);
                acc[m][a][1] = fmaf(x, s.y, acc[m][a][1]);
                acc[m][a][2] = fmaf(x, s.z, acc[m][a][2]);
                acc[m][a][3] = fmaf(x, s.w, acc[m][a][3]);
            }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = row0 + r0 + a;
            if (i < B) {
                float *dst = (m ? qs0 : ks0) + (((size_t)b * B + i) * H + h) * kGdnD + c0;
                *reinterpret_cast<float4 *>(dst) = make_float4(acc[m][a][0], acc[m][a][1], acc[m][a][2], acc[m][a][3]);
            }
        }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kGdnThreads) gdn_tree_solve_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const float *__restrict__ alpha, const float *__restrict__ beta, const int32_t *__restrict__ parent,
    const float *__restrict__ ks0, const float *__restrict__ qs0, int B, int H, float *__restrict__ O,
    int32_t *status)
{
    extern __shared__ float4 gdn_smem[];
    float *s_u = reinterpret_cast<float *>(gdn_smem);                 // [B][D] u_i
    uint16_t *s_k = reinterpret_cast<uint16_t *>(s_u + (size_t)B * kGdnD);  // [B][D] k_i (bf16)
    float *s_gamma = reinterpret_cast<float *>(s_k + (size_t)B * kGdnD);    // [B]
    float *s_alpha = s_gamma + B;                                            // [B]
    int *s_parent = reinterpret_cast<int *>(s_alpha + B);                   // [B]
    volatile int *s_done = s_parent + B;                                     // [B]
    __shared__ int s_abort;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nwarps = kGdnThreads / 32;

    // inputs that do not come from the dense kernel
    bool bad = false;
    for (int i = tid; i < B; i += kGdnThreads) {
        const int p = parent[(size_t)b * B + i];
        bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
        s_parent[i] = p;
        s_alpha[i] = alpha[((size_t)b * B + i) * H + h];
        s_done[i] = 0;
    }
    for (int t = tid; t < B * kGdnD / 8; t += kGdnThreads) {
        const int i = t / (kGdnD / 8), d8 = t - i * (kGdnD / 8);
        reinterpret_cast<uint4 *>(s_k)[t] =
            reinterpret_cast<const uint4 *>(k + (((size_t)b * B + i) * H + h) * kGdnD)[d8];
    }
    if (tid == 0) s_abort = 0;
    const bool any_bad = __syncthreads_or(bad);
    pdl_wait_primary();  // K S0 and Q S0 come from the dense kernel (waited even on bad input)
    if (any_bad) {
        if (tid == 0) report_status(status, TV_ERR_NOT_TOPOLOGICAL);
        return;
    }

    for (int i = wid; i < B; i += nwarps) {
        const int p = s_parent[i];
        // wait (bounded) until the parent is done: then all ancestors are
        if (p >= 0) {
            const uint64_t t0 = global_timer_ns();
            bool ok = true;
            for (uint32_t it = 0; s_done[p] == 0; ++it) {
                if ((it & 63) == 63 && (s_abort || global_timer_ns() - t0 > kWaitLimitNs)) {
                    ok = false;
                    break;
                }
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    s_abort = 1;
                    report_status(status, TV_ERR_TIMEOUT);
                }
                break;
            }
            __threadfence_block();  // the ancestors' u rows are visible from here
        }
        const size_t row = ((size_t)b * B + i) * H + h;
        const float ai = s_alpha[i], bi = beta[row];
        const float gi = (p >= 0 ? s_gamma[p] : 1.f) * ai;
        // lane l holds columns 4l .. 4l+3 of this node's vectors
        float ki[4], qi[4], acc_u[4] = {0.f, 0.f, 0.f, 0.f}, acc_o[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint2 kk = reinterpret_cast<const uint2 *>(s_k + (size_t)i * kGdnD)[lane];
            const uint2 qq = reinterpret_cast<const uint2 *>(q + row * kGdnD)[lane];
            ki[0] = bf16_to_f32(kk.x & 0xFFFFu); ki[1] = bf16_to_f32(kk.x >> 16);
            ki[2] = bf16_to_f32(kk.y & 0xFFFFu); ki[3] = bf16_to_f32(kk.y >> 16);
            qi[0] = bf16_to_f32(qq.x & 0xFFFFu); qi[1] = bf16_to_f32(qq.x >> 16);
            qi[2] = bf16_to_f32(qq.y & 0xFFFFu); qi[3] = bf16_to_f32(qq.y >> 16);
        }
        // strict ancestors j = p, parent(p), ...: r = gamma_i / gamma_j as a running product
        float r = ai;
        for (int j = p; j >= 0; j = s_parent[j]) {
            const uint2 kk = reinterpret_cast<const uint2 *>(s_k + (size_t)j * kGdnD)[lane];
            const float k0 = bf16_to_f32(kk.x & 0xFFFFu), k1 = bf16_to_f32(kk.x >> 16);
            const float k2 = bf16_to_f32(kk.y & 0xFFFFu), k3 = bf16_to_f32(kk.y >> 16);
            const float g = warp_sum(ki[0] * k0 + ki[1] * k1 + ki[2] * k2 + ki[3] * k3) * r;
            const float a = warp_sum(qi[0] * k0 + qi[1] * k1 + qi[2] * k2 + qi[3] * k3) * r;
            const float4 uj = reinterpret_cast<const float4 *>(s_u + (size_t)j * kGdnD)[lane];
            acc_u[0] = fmaf(g, uj.x, acc_u[0]); acc_u[1] = fmaf(g, uj.y, acc_u[1]);
            acc_u[2] = fmaf(g, uj.z, acc_u[2]); acc_u[3] = fmaf(g, uj.w, acc_u[3]);
            acc_o[0] = fmaf(a, uj.x, acc_o[0]); acc_o[1] = fmaf(a, uj.y, acc_o[1]);
            acc_o[2] = fmaf(a, uj.z, acc_o[2]); acc_o[3] = fmaf(a, uj.w, acc_o[3]);
            r *= s_alpha[j];
        }
        const float4 ks = reinterpret_cast<const float4 *>(ks0 + row * kGdnD)[lane];
        const float4 qs = reinterpret_cast<const float4 *>(qs0 + row * kGdnD)[lane];
        const uint2 vv = reinterpret_cast<const uint2 *>(v + row * kGdnD)[lane];
        const float vi[4] = {bf16_to_f32(vv.x & 0xFFFFu), bf16_to_f32(vv.x >> 16), bf16_to_f32(vv.y & 0xFFFFu),
                             bf16_to_f32(vv.y >> 16)};
        const float ksv[4] = {ks.x, ks.y, ks.z, ks.w}, qsv[4] = {qs.x, qs.y, qs.z, qs.w};
        float ui[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) ui[c] = bi * (vi[c] - gi * ksv[c] - acc_u[c]);
        const float aii = warp_sum(qi[0] * ki[0] + qi[1] * ki[1] + qi[2] * ki[2] + qi[3] * ki[3]);
        reinterpret_cast<float4 *>(s_u + (size_t)i * kGdnD)[lane] = make_float4(ui[0], ui[1], ui[2], ui[3]);
        if (lane == 0) s_gamma[i] = gi;
        float4 o;
        o.x = gi * qsv[0] + acc_o[0] + aii * ui[0];
        o.y = gi * qsv[1] + acc_o[1] + aii * ui[1];
        o.z = gi * qsv[2] + acc_o[2] + aii * ui[2];
        o.w = gi * qsv[3] + acc_o[3] + aii * ui[3];
        reinterpret_cast<float4 *>(O + row * kGdnD)[lane] = o;
        __threadfence_block();  // every lane's u_i (and gamma_i) before the done flag
        __syncwarp();
        if (lane == 0) s_done[i] = 1;
    }
}

size_t gdn_workspace_bytes(int nb, int B, int H) { return (size_t)2 * nb * B * H * kGdnD * sizeof(float); }

static size_t gdn_solve_smem(int B)
{
    return (size_t)B * kGdnD * (sizeof(float) + sizeof(uint16_t)) + (size_t)B * (2 * sizeof(float) + 2 * sizeof(int));
}

cudaError_t launch_gdn_tree(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                            const float *beta, const float *S0, const int32_t *parent, int nb, int B, int H, float *O,
                            void *workspace, int32_t *status, cudaStream_t stream)
{
    static int opted_in[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem1 = (size_t)kGdnD * kGdnD * sizeof(float) + (size_t)2 * kGdnRows * kGdnD * sizeof(float);
    if (!(dev >= 0 && dev < 64 && opted_in[dev])) {
        e = cudaFuncSetAttribute(gdn_state_products_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gdn_tree_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)gdn_solve_smem(kGdnMaxB));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = 1;
    }
    float *ks0 = static_cast<float *>(workspace);
    float *qs0 = ks0 + (size_t)nb * B * H * kGdnD;
    e = launch_dependent(gdn_state_products_kernel, dim3((unsigned)((B + kGdnRows - 1) / kGdnRows), (unsigned)H,
                                                         (unsigned)nb),
                         dim3(kGdnThreads), smem1, stream, q, k, S0, B, H, ks0, qs0);
    if (e != cudaSuccess) return e;
    return launch_dependent(gdn_tree_solve_kernel, dim3((unsigned)H, (unsigned)nb), dim3(kGdnThreads),
                            gdn_solve_smem(B), stream, q, k, v, alpha, beta, parent, (const float *)ks0,
                            (const float *)qs0, B, H, O, status);
}

}  // namespace tv
