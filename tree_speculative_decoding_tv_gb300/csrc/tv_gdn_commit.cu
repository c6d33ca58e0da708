// Commit of a Gated DeltaNet layer's state for the accepted branch.
//
// DFlash-TfM summary, §3 "Verificación de Árboles sin Rollback": tree verification
// leaves the committed state S0 untouched, and the state is committed in the next
// decoding iteration, once the accepted branch is known, so nothing is rolled back.
// Committing is the recurrence
//   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
// applied from S0 to the accepted root path path[0] (the root) .. path[n_acc] in
// order.  With w = k^T S_{t-1} (one value per state column), one step is
//   S_t = alpha S_{t-1} + k (beta (v - alpha w))^T.
//
// GPU form.  A state column evolves on its own: w_c and the update of column c use
// column c alone.  So one warp takes 4 columns of one head, lane l holding column
// l % 4 for 16 contiguous key rows 16 (l / 4) .. +15 in registers; 4 warps (16
// columns) make a CTA, and the D / 16 CTAs of a head run side by side.  The path's
// k rows, its v entries for the CTA's columns and its gates are staged in shared
// memory in one round trip.  A step is then warp-local: 16 fused multiply-adds, a
// 3-level shuffle sum over the row groups, and 16 updates; no barrier.  S_out may be
// S0 itself: every lane reads exactly the entries it writes, before writing them.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kCommitD = 128;
constexpr int kCommitCols = 4;                                 // state columns per warp
constexpr int kCommitWarps = 4;                                // warps per CTA
constexpr int kCommitThreads = 32 * kCommitWarps;
constexpr int kCommitCtaCols = kCommitCols * kCommitWarps;     // 16 columns per CTA
constexpr int kCommitRows = kCommitD / (32 / kCommitCols);     // 16 key rows per lane
static_assert(kCommitRows == 16 && kCommitD % kCommitCtaCols == 0, "row split");

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__global__ void __launch_bounds__(kCommitThreads) gdn_commit_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, const float *__restrict__ alpha,
    const float *__restrict__ beta, const float *S0, const int32_t *__restrict__ n_acc,
    const int32_t *__restrict__ path, int B, int H, float *S_out, int32_t *status)
{
    extern __shared__ uint4 gc_smem[];
    uint16_t *s_k = reinterpret_cast<uint16_t *>(gc_smem);  // [B][D] path order
    uint16_t *s_v = s_k + (size_t)B * kCommitD;              // [B][16] this CTA's columns
    float *s_a = reinterpret_cast<float *>(s_v + (size_t)B * kCommitCtaCols);  // [B]
    float *s_b = s_a + B;                                                      // [B]
    const int h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x, lane = tid & 31;
    const int col0 = blockIdx.x * kCommitCtaCols;
    const int cl = (tid >> 5) * kCommitCols + (lane & (kCommitCols - 1));  // column inside the CTA's 16
    const int c = col0 + cl, r0 = (lane / kCommitCols) * kCommitRows;
    const size_t bh = (size_t)b * H + h;

    pdl_wait_primary();  // n_acc and path come from the acceptance kernel
    pdl_launch_dependents();
    // this lane's state entries (read before anything is written: S_out may be S0)
    const float *src = S0 + bh * kCommitD * kCommitD;
    float S[kCommitRows];
#pragma unroll
    for (int e = 0; e < kCommitRows; ++e) S[e] = src[(size_t)(r0 + e) * kCommitD + c];
    const int n = n_acc[b];
    const int32_t *pr = path + (size_t)b * B;
    // the path: root first, strictly increasing, inside the tree
    bool bad = n < 0 || n >= B;
    if (!bad)
        for (int t = tid; t <= n; t += kCommitThreads) {
            const int p = pr[t];
            if (t == 0 ? p != 0 : (p <= pr[t - 1] || p >= B)) bad = true;
        }
    const bool any_bad = __syncthreads_or(bad);
    float *dst = S_out + bh * kCommitD * kCommitD;
    if (any_bad) {  // nothing is committed
        if (tid == 0 && h == 0 && blockIdx.x == 0) report_status(status, TV_ERR_INVALID_ARG);
#pragma unroll
        for (int e = 0; e < kCommitRows; ++e) dst[(size_t)(r0 + e) * kCommitD + c] = S[e];
        return;
    }

    // stage the path's k rows, v entries and gates (all loads in flight together)
    const int len = n + 1;
    constexpr int kQk = kCommitD / 8, kQv = kCommitCtaCols / 8;  // 16-byte pieces per k row, per v slice
    for (int idx = tid; idx < len * (kQk + kQv); idx += kCommitThreads) {
        const int t = idx / (kQk + kQv), q = idx - t * (kQk + kQv);
        const size_t row = ((size_t)b * B + pr[t]) * H + h;
        if (q < kQk)
            reinterpret_cast<uint4 *>(s_k + (size_t)t * kCommitD)[q] = reinterpret_cast<const uint4 *>(k + row * kCommitD)[q];
        else
            reinterpret_cast<uint4 *>(s_v + (size_t)t * kCommitCtaCols)[q - kQk] =
                reinterpret_cast<const uint4 *>(v + row * kCommitD + col0)[q - kQk];
    }
    for (int t = tid; t < len; t += kCommitThreads) {
        const size_t row = ((size_t)b * B + pr[t]) * H + h;
        s_a[t] = alpha[row];
        s_b[t] = beta[row];
    }
    __syncthreads();

    for (int t = 0; t < len; ++t) {
        const uint4 *kq = reinterpret_cast<const uint4 *>(s_k + (size_t)t * kCommitD + r0);
        const uint4 k0 = kq[0], k1 = kq[1];
        const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        float kf[kCommitRows];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kf[2 * e] = bf16_lo(kw[e]);  // the lower address holds the lower half
            kf[2 * e + 1] = bf16_hi(kw[e]);
        }
        float w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < kCommitRows; ++e) w4[e & 3] = fmaf(kf[e], S[e], w4[e & 3]);
        float w = (w4[0] + w4[1]) + (w4[2] + w4[3]);
#pragma unroll
        for (int o = kCommitCols; o < 32; o <<= 1) w += __shfl_xor_sync(0xffffffffu, w, o);  // over row groups
        const float a = s_a[t], be = s_b[t];
        const float coef = be * (bf16f(s_v[(size_t)t * kCommitCtaCols + cl]) - a * w);
#pragma unroll
        for (int e = 0; e < kCommitRows; ++e) S[e] = fmaf(kf[e], coef, a * S[e]);
    }
#pragma unroll
    for (int e = 0; e < kCommitRows; ++e) dst[(size_t)(r0 + e) * kCommitD + c] = S[e];
}

size_t gdn_commit_smem_bytes(int B) { return (size_t)B * (kCommitD * 2 + kCommitCtaCols * 2 + 2 * 4); }

cudaError_t launch_gdn_commit(const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                              const float *S0, const int32_t *n_acc, const int32_t *path, int nb, int B, int H,
                              float *S_out, int32_t *status, cudaStream_t stream)
{
    static int opted_in[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!(dev >= 0 && dev < 64 && opted_in[dev])) {
        e = cudaFuncSetAttribute(gdn_commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)gdn_commit_smem_bytes(256));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = 1;
    }
    return launch_dependent(gdn_commit_kernel, dim3((unsigned)(kCommitD / kCommitCtaCols), (unsigned)H, (unsigned)nb),
                            dim3(kCommitThreads), gdn_commit_smem_bytes(B), stream, k, v, alpha, beta, S0, n_acc,
                            path, B, H, S_out, status);
}

}  // namespace tv
