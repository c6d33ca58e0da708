// Commit of the accepted branch's K/V into the paged cache.
//
// The pages commit state only once the accepted branch is known (DFlash-TfM
// summary, §3 "Solución"), so nothing is rolled back.  For attention the state is
// the paged K/V cache: sequence b holds its committed tokens at logical positions
// [0, P) (P = prefix_lens[b]) and tree node t at P + t.  The commit keeps the root
// and the accepted nodes in path order: position P + k takes what P + path[b][k]
// held, for k = 1 .. n_acc[b] (the root stays at P), and the committed length
// becomes P + n_acc[b] + 1.
//
// GPU form: one CTA per (sequence, kv head).  A source row can be another row's
// destination (path 0, 1, 3, 5 moves 3 -> 2 and 5 -> 3), so the CTA first stages
// every row that moves (K and V, 256 bytes each at D = 128) in shared memory with
// 16-byte loads, synchronises, then writes them.  Rows already in place
// (path[k] == k) are skipped.  The work is a few kilobytes per sequence: the
// kernel is latency-bound, and it reads nothing before the previous kernel (the
// acceptance, which produces n_acc and path) has completed.
#include <cuda_runtime.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kCommitThreads = 256;
constexpr int kCommitMaxB = 256;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(uint16_t *__restrict__ k_cache,
                                                                   uint16_t *__restrict__ v_cache,
                                                                   const int32_t *__restrict__ block_table,
                                                                   const int32_t *__restrict__ prefix_lens,
                                                                   const int32_t *__restrict__ n_acc,
                                                                   const int32_t *__restrict__ path, int B, int Hkv,
                                                                   int D, int num_blocks, int max_pages,
                                                                   int32_t *__restrict__ new_prefix_lens,
                                                                   int32_t *status)
{
    extern __shared__ uint4 stage[];  // [moving rows][K, V][D / 8] 16-byte vectors
    __shared__ int s_src[kCommitMaxB], s_dst[kCommitMaxB];
    __shared__ int s_count;
    const int b = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
    const int page = 16;
    const int vecs = D / 8;  // 16-byte vectors per row

    pdl_wait_primary();  // n_acc and path come from the previous kernel; earlier readers of the caches are done
    pdl_launch_dependents();
    const int P = prefix_lens[b];
    const int n = n_acc[b];
    const int32_t *pr = path + (size_t)b * B;
    const int32_t *bt = block_table + (size_t)b * max_pages;

    // validation: a root path of at most B nodes, every touched position inside the block table
    bool bad = P < 0 || n < 0 || n >= B || (long long)P + B > (long long)max_pages * page;
    int src_row = -1, dst_row = -1;  // physical row index (block * Hkv + g) * 16 + slot, for k = tid
    const int k = tid;
    if (!bad && k <= n) {  // k = 0 is the root: checked, never moved
        const int pk = pr[k];
        if (k == 0 ? pk != 0 : (pk <= pr[k - 1] || pk >= B)) {
            bad = true;
        } else {
            const int xs = P + pk, xd = P + k;
            const int bs = bt[xs / page], bd = bt[xd / page];
            if (bs < 0 || bs >= num_blocks || bd < 0 || bd >= num_blocks) {
                bad = true;
            } else if (pk != k) {
                src_row = (bs * Hkv + g) * page + xs % page;
                dst_row = (bd * Hkv + g) * page + xd % page;
            }
        }
    }
    if (tid == 0) s_count = 0;
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            report_status(status, TV_ERR_INVALID_ARG);
            if (g == 0) new_prefix_lens[b] = P;  // nothing committed
        }
        return;
    }
    if (src_row >= 0) {  // compact the rows that move
        const int slot = atomicAdd(&s_count, 1);
        s_src[slot] = src_row;
        s_dst[slot] = dst_row;
    }
    __syncthreads();
    const int m = s_count;
    const int per_row = 2 * vecs;  // K then V
    for (int t = tid; t < m * per_row; t += kCommitThreads) {
        const int r = t / per_row, c = t - r * per_row;
        const uint16_t *cache = c < vecs ? k_cache : v_cache;
        stage[t] = reinterpret_cast<const uint4 *>(cache + (size_t)s_src[r] * D)[c % vecs];
    }
    __syncthreads();
    for (int t = tid; t < m * per_row; t += kCommitThreads) {
        const int r = t / per_row, c = t - r * per_row;
        uint16_t *cache = c < vecs ? k_cache : v_cache;
        reinterpret_cast<uint4 *>(cache + (size_t)s_dst[r] * D)[c % vecs] = stage[t];
    }
    if (tid == 0 && g == 0) new_prefix_lens[b] = P + n + 1;
}

size_t kv_commit_smem_bytes(int B, int D) { return (size_t)(B - 1) * 2 * D * sizeof(uint16_t); }

cudaError_t launch_kv_commit(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_table,
                             const int32_t *prefix_lens, const int32_t *n_acc, const int32_t *path, int nb, int B,
                             int Hkv, int D, int num_blocks, int max_pages, int32_t *new_prefix_lens, int32_t *status,
                             cudaStream_t stream)
{
    static int opted_in[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = kv_commit_smem_bytes(B, D);
    if (smem > 48 * 1024 && !(dev >= 0 && dev < 64 && opted_in[dev])) {
        e = cudaFuncSetAttribute(kv_commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kv_commit_smem_bytes(kCommitMaxB, 128));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) opted_in[dev] = 1;
    }
    return launch_dependent(kv_commit_kernel, dim3((unsigned)nb, (unsigned)Hkv), dim3(kCommitThreads), smem, stream,
                            k_cache, v_cache, block_table, prefix_lens, n_acc, path, B, Hkv, D, num_blocks, max_pages,
                            new_prefix_lens, status);
}

}  // namespace tv
