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
// GPU form: one 256-thread CTA per (sequence, head).  Thread t holds column
// c = t % 128 of the state for key rows 64 (t / 128) .. +63 in registers.  The
// path's k and v rows (bf16) and gates are staged in shared memory in one round
// trip; each step is then a column sum over the thread's 64 rows, one barrier to
// add the two halves (double-buffered, so one barrier per step), and 64 fused
// multiply-adds.  S_out may be S0 itself: every thread reads its entries before
// any is written.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kCommitD = 128;
constexpr int kCommitThreads = 256;
constexpr int kCommitRows = kCommitD / 2;  // key rows per thread: two threads per state column
static_assert(2 * kCommitD == kCommitThreads, "two threads per state column");

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__global__ void __launch_bounds__(kCommitThreads) gdn_commit_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, const float *__restrict__ alpha,
    const float *__restrict__ beta, const float *S0, const int32_t *__restrict__ n_acc,
    const int32_t *__restrict__ path, int B, int H, float *S_out, int32_t *status)
{
    extern __shared__ uint4 gc_smem[];
    uint16_t *s_k = reinterpret_cast<uint16_t *>(gc_smem);  // [B][D] path order
    uint16_t *s_v = s_k + (size_t)B * kCommitD;              // [B][D]
    float *s_a = reinterpret_cast<float *>(s_v + (size_t)B * kCommitD);  // [B]
    float *s_b = s_a + B;                                                // [B]
    __shared__ float s_w[2][2][kCommitD];  // [step parity][half][column]
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int c = tid & (kCommitD - 1), half = tid >> 7;
    const size_t bh = (size_t)b * H + h;

    pdl_wait_primary();  // n_acc and path come from the acceptance kernel
    pdl_launch_dependents();
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

    // this thread's state entries (read before anything is written: S_out may be S0)
    const float *src = S0 + bh * kCommitD * kCommitD;
    float S[kCommitRows];
#pragma unroll
    for (int e = 0; e < kCommitRows; ++e) S[e] = src[(size_t)(half * kCommitRows + e) * kCommitD + c];
    float *dst = S_out + bh * kCommitD * kCommitD;
    if (any_bad) {  // nothing is committed
        if (tid == 0 && h == 0) report_status(status, TV_ERR_INVALID_ARG);
        __syncthreads();
#pragma unroll
        for (int e = 0; e < kCommitRows; ++e) dst[(size_t)(half * kCommitRows + e) * kCommitD + c] = S[e];
        return;
    }

    // stage the path's rows and gates (all loads in flight together)
    const int len = n + 1;
    for (int idx = tid; idx < 2 * len * (kCommitD / 8); idx += kCommitThreads) {
        const int which = idx / (len * (kCommitD / 8)), rem = idx - which * len * (kCommitD / 8);
        const int t = rem / (kCommitD / 8), q = rem - t * (kCommitD / 8);
        const size_t row = ((size_t)b * B + pr[t]) * H + h;
        reinterpret_cast<uint4 *>((which ? s_v : s_k) + (size_t)t * kCommitD)[q] =
            reinterpret_cast<const uint4 *>((which ? v : k) + row * kCommitD)[q];
    }
    for (int t = tid; t < len; t += kCommitThreads) {
        const size_t row = ((size_t)b * B + pr[t]) * H + h;
        s_a[t] = alpha[row];
        s_b[t] = beta[row];
    }
    __syncthreads();

    for (int t = 0; t < len; ++t) {
        const uint16_t *kt = s_k + (size_t)t * kCommitD + half * kCommitRows;
        float w = 0.f;
#pragma unroll
        for (int e = 0; e < kCommitRows; ++e) w = fmaf(bf16f(kt[e]), S[e], w);
        s_w[t & 1][half][c] = w;
        __syncthreads();  // (the other parity's buffer is free: everyone passed the previous barrier)
        const float a = s_a[t], be = s_b[t];
        const float wc = s_w[t & 1][0][c] + s_w[t & 1][1][c];
        const float coef = be * (bf16f(s_v[(size_t)t * kCommitD + c]) - a * wc);
#pragma unroll
        for (int e = 0; e < kCommitRows; ++e) S[e] = fmaf(bf16f(kt[e]), coef, a * S[e]);
    }
#pragma unroll
    for (int e = 0; e < kCommitRows; ++e) dst[(size_t)(half * kCommitRows + e) * kCommitD + c] = S[e];
}

size_t gdn_commit_smem_bytes(int B) { return (size_t)B * (2 * kCommitD * 2 + 2 * 4); }

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
    return launch_dependent(gdn_commit_kernel, dim3((unsigned)H, (unsigned)nb), dim3(kCommitThreads),
                            gdn_commit_smem_bytes(B), stream, k, v, alpha, beta, S0, n_acc, path, B, H, S_out,
                            status);
}

}  // namespace tv
