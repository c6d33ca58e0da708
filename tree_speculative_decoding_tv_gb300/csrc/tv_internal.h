// Internal launch interface between the C ABI (tv_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/treeverify.h"

namespace tv {

// Launch `kernel` on `stream` as a programmatic dependent of the stream's previous
// kernel: it may be scheduled while that kernel drains, and must execute
// griddepcontrol.wait (pdl_wait_primary) before reading anything that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_build_mask(const int32_t *parent, int B, int nb, uint32_t *mask, int32_t *depth, int32_t *status,
                              cudaStream_t stream);

// Workspace bytes tv_accept needs: one 8-byte partial per (row, 8192-logit chunk).
size_t accept_workspace_bytes(int V, int B, int nb);

cudaError_t launch_accept(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                          const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                          int32_t *bonus, int32_t *status, void *workspace, int num_sms, cudaStream_t stream);

// Workspace bytes tv_accept_fused needs: the keys, then one 32-bit counter per sequence.
size_t accept_fused_workspace_bytes(int V, int B, int nb);

// Argmax and acceptance in one kernel; mask may be null.
cudaError_t launch_accept_fused(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                                const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                                int32_t *bonus, int32_t *status, void *workspace, int num_sms, cudaStream_t stream);

// tv_accept on the library's own static scratch (no workspace argument).
cudaError_t launch_accept_noalloc(const uint16_t *logits, int V, const int32_t *draft, const int32_t *parent,
                                  const uint32_t *mask, int B, int nb, int32_t *am, int32_t *n_acc, int32_t *path,
                                  int32_t *bonus, int32_t *status, int num_sms, cudaStream_t stream);

// Best-first draft-tree construction with top-w rounds (one warp per sequence).
cudaError_t launch_build_tree(const float *logp, const int32_t *tok, int nb, int Dmax, int K, int B, int w,
                              int32_t *parent, int32_t *token, float *score, int32_t *status, cudaStream_t stream);

// Gated DeltaNet tree verification: dense K S0 / Q S0 products, then the sparse
// masked solve and outputs (4 CTAs per (sequence, head), one per 32 value columns).
size_t gdn_workspace_bytes(int nb, int B, int H);
cudaError_t launch_gdn_tree(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                            const float *beta, const float *S0, const int32_t *parent, int nb, int B, int H, float *O,
                            void *workspace, int32_t *status, cudaStream_t stream);

// Gated DeltaNet state commit along the accepted path (8 CTAs per (sequence, head), one
// per 16 state columns).
cudaError_t launch_gdn_commit(const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                              const float *S0, const int32_t *n_acc, const int32_t *path, int nb, int B, int H,
                              float *S_out, int32_t *status, cudaStream_t stream);

// Commit of the accepted branch's K/V (one CTA per (sequence, kv head)).
cudaError_t launch_kv_commit(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_table,
                             const int32_t *prefix_lens, const int32_t *n_acc, const int32_t *path, int nb, int B,
                             int Hkv, int D, int num_blocks, int max_pages, int32_t *new_prefix_lens, int32_t *status,
                             cudaStream_t stream);

// A kernel whose only job is to take the bounded-wait timeout path (see tv_selftest.cu).
cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t *status, cudaStream_t stream);

// Workspace bytes the attention needs with `ctas` CTAs over `row_tiles`
// (sequence, kv head, 128-row tile) units, and that unit count for `a`.
size_t attn_workspace_bytes(int ctas, int row_tiles);
int attn_row_tiles(const tv_attn_args *a);
// Kernels launch_attn enqueues for `a` with `ctas` CTAs: 1, or 2 with the merge kernel.
int attn_kernel_launches(const tv_attn_args *a, int ctas);

// Encodes the TMA descriptors and launches the attention kernel and its merge kernel.
// Returns TV_OK or TV_ERR_CUDA (with *cuda_err set).
int32_t launch_attn(const tv_attn_args *a, int ctas, void *workspace, cudaStream_t stream, cudaError_t *cuda_err);

}  // namespace tv
