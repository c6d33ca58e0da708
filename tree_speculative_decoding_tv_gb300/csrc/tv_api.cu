// C ABI of libtreeverify: argument validation and kernel dispatch.
// Entry points and their contracts are declared and documented in
// include/treeverify.h.
#include <cuda_runtime.h>

#include <cstdint>

#include "tv_internal.h"

namespace {

constexpr int kMaxB = 256;
constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool group_supported(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// Validates everything about tv_attn_args that can be checked on the host.
int32_t check_attn(const tv_attn_args *a)
{
    if (!a) return TV_ERR_INVALID_ARG;
    if (a->nb < 0) return TV_ERR_INVALID_ARG;
    if (a->B < 1 || a->B > kMaxB) return TV_ERR_UNSUPPORTED_SHAPE;
    if (a->D != kHeadDim || a->page_size != kPageSize) return TV_ERR_UNSUPPORTED_SHAPE;
    if (a->Hq < 1 || a->Hkv < 1 || a->Hq % a->Hkv != 0) return TV_ERR_INVALID_ARG;
    if (!group_supported(a->Hq / a->Hkv)) return TV_ERR_UNSUPPORTED_SHAPE;
    if (a->num_blocks < 1 || a->max_pages < 1) return TV_ERR_INVALID_ARG;
    if ((long long)a->max_pages * kPageSize >= (1ll << 30)) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)a->num_blocks * a->Hkv * kPageSize >= (1ll << 31)) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)a->nb * a->B * a->Hq >= (1ll << 31)) return TV_ERR_UNSUPPORTED_SHAPE;
    if (a->num_ctas < 0) return TV_ERR_INVALID_ARG;
    if (!a->q_d || !a->k_cache_d || !a->v_cache_d || !a->block_table_d || !a->prefix_lens_d ||
        (!a->mask_d && !a->parent_d) || !a->o_d || !a->lse_d)
        return TV_ERR_INVALID_ARG;
    if (!aligned(a->q_d, 16) || !aligned(a->k_cache_d, 16) || !aligned(a->v_cache_d, 16) || !aligned(a->o_d, 16))
        return TV_ERR_INVALID_ARG;
    if (!aligned(a->block_table_d, 4) || !aligned(a->prefix_lens_d, 4) || !aligned(a->mask_d, 4) ||
        !aligned(a->parent_d, 4) || !aligned(a->lse_d, 4) || !aligned(a->dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    return TV_OK;
}

// The acceptance kernels index a row with 32-bit ints and cut it into 4096-logit
// units: V and the unit count must stay clear of 2^31.
bool accept_shape_ok(int32_t V, int32_t B, int32_t nb)
{
    if ((long long)V > (long long)INT32_MAX - 8192) return false;
    return (long long)nb * B * (((long long)V + 4095) / 4096) < (1ll << 31);
}

int attn_ctas(const tv_attn_args *a)
{
    if (a->num_ctas > 0) return a->num_ctas;
    return sm_count();
}

}  // namespace

extern "C" {

const char *tv_status_str(int32_t s)
{
    switch (s) {
    case TV_OK: return "TV_OK";
    case TV_ERR_INVALID_ARG: return "TV_ERR_INVALID_ARG";
    case TV_ERR_NOT_TOPOLOGICAL: return "TV_ERR_NOT_TOPOLOGICAL";
    case TV_ERR_UNSUPPORTED_SHAPE: return "TV_ERR_UNSUPPORTED_SHAPE";
    case TV_ERR_CUDA: return "TV_ERR_CUDA";
    case TV_ERR_TIMEOUT: return "TV_ERR_TIMEOUT";
    case TV_ERR_UNIMPLEMENTED: return "TV_ERR_UNIMPLEMENTED";
    default: return "TV_ERR_UNKNOWN";
    }
}

int32_t tv_version(void) { return 100; }

int32_t tv_build_mask(const int32_t *parent_d, int32_t B, int32_t nb, uint32_t *mask_d, int32_t *depth_d,
                      int32_t *dev_status_d, void *stream)
{
    if (nb < 0) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return TV_ERR_UNSUPPORTED_SHAPE;
    if (!parent_d || !mask_d) return TV_ERR_INVALID_ARG;
    if (!aligned(parent_d, 4) || !aligned(mask_d, 4) || !aligned(depth_d, 4) || !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (nb == 0) return TV_OK;
    cudaError_t e = tv::launch_build_mask(parent_d, B, nb, mask_d, depth_d, dev_status_d,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

size_t tv_attn_workspace_size(const tv_attn_args *args)
{
    if (check_attn(args) != TV_OK) return 0;
    const int ctas = attn_ctas(args);
    if (ctas < 1) return 0;
    return tv::attn_workspace_bytes(ctas, tv::attn_row_tiles(args));
}

int32_t tv_attn_launches(const tv_attn_args *args)
{
    if (check_attn(args) != TV_OK || args->nb == 0) return 0;
    const int ctas = attn_ctas(args);
    if (ctas < 1) return 0;
    return tv::attn_kernel_launches(args, ctas);
}

int32_t tv_attn(const tv_attn_args *args, void *workspace_d, size_t workspace_bytes, void *stream)
{
    const int32_t rc = check_attn(args);
    if (rc != TV_OK) return rc;
    if (args->nb == 0) return TV_OK;
    const int ctas = attn_ctas(args);
    if (ctas < 1) return TV_ERR_CUDA;
    if (!workspace_d || !aligned(workspace_d, 16) || workspace_bytes < tv::attn_workspace_bytes(ctas, tv::attn_row_tiles(args)))
        return TV_ERR_INVALID_ARG;
    cudaError_t e;
    return tv::launch_attn(args, ctas, workspace_d, static_cast<cudaStream_t>(stream), &e);
}

size_t tv_accept_workspace_size(int32_t V, int32_t B, int32_t nb)
{
    if (V < 1 || B < 1 || B > kMaxB || nb < 0) return 0;
    return tv::accept_workspace_bytes(V, B, nb);
}

int32_t tv_accept(const uint16_t *logits_d, int32_t V, const int32_t *draft_tokens_d, const int32_t *parent_d,
                  const uint32_t *mask_d, int32_t B, int32_t nb, int32_t *argmax_d, int32_t *n_acc_d,
                  int32_t *path_d, int32_t *bonus_d, int32_t *dev_status_d, void *workspace_d,
                  size_t workspace_bytes, void *stream)
{
    if (nb < 0 || V < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return TV_ERR_UNSUPPORTED_SHAPE;
    if (!logits_d || !draft_tokens_d || !parent_d || !argmax_d || !n_acc_d || !path_d || !bonus_d)
        return TV_ERR_INVALID_ARG;
    if (!aligned(logits_d, 2) || !aligned(draft_tokens_d, 4) || !aligned(parent_d, 4) || !aligned(mask_d, 4) ||
        !aligned(argmax_d, 4) || !aligned(n_acc_d, 4) || !aligned(path_d, 4) || !aligned(bonus_d, 4) ||
        !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (!accept_shape_ok(V, B, nb)) return TV_ERR_UNSUPPORTED_SHAPE;
    if (nb == 0) return TV_OK;
    if (!workspace_d || !aligned(workspace_d, 8) || workspace_bytes < tv::accept_workspace_bytes(V, B, nb))
        return TV_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms < 1) return TV_ERR_CUDA;
    cudaError_t e = tv::launch_accept(logits_d, V, draft_tokens_d, parent_d, mask_d, B, nb, argmax_d, n_acc_d,
                                      path_d, bonus_d, dev_status_d, workspace_d, sms,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

size_t tv_accept_fused_workspace_size(int32_t V, int32_t B, int32_t nb)
{
    if (V < 1 || B < 1 || B > kMaxB || nb < 0) return 0;
    return tv::accept_fused_workspace_bytes(V, B, nb);
}

int32_t tv_accept_fused(const uint16_t *logits_d, int32_t V, const int32_t *draft_tokens_d, const int32_t *parent_d,
                        const uint32_t *mask_d, int32_t B, int32_t nb, int32_t *argmax_d, int32_t *n_acc_d,
                        int32_t *path_d, int32_t *bonus_d, int32_t *dev_status_d, void *workspace_d,
                        size_t workspace_bytes, void *stream)
{
    if (nb < 0 || V < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return TV_ERR_UNSUPPORTED_SHAPE;
    if (!logits_d || !draft_tokens_d || !parent_d || !argmax_d || !n_acc_d || !path_d || !bonus_d)
        return TV_ERR_INVALID_ARG;
    if (!aligned(logits_d, 2) || !aligned(draft_tokens_d, 4) || !aligned(parent_d, 4) || !aligned(mask_d, 4) ||
        !aligned(argmax_d, 4) || !aligned(n_acc_d, 4) || !aligned(path_d, 4) || !aligned(bonus_d, 4) ||
        !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (!accept_shape_ok(V, B, nb)) return TV_ERR_UNSUPPORTED_SHAPE;
    if (nb == 0) return TV_OK;
    if (!workspace_d || !aligned(workspace_d, 8) || workspace_bytes < tv::accept_fused_workspace_bytes(V, B, nb))
        return TV_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms < 1) return TV_ERR_CUDA;
    cudaError_t e = tv::launch_accept_fused(logits_d, V, draft_tokens_d, parent_d, mask_d, B, nb, argmax_d, n_acc_d,
                                            path_d, bonus_d, dev_status_d, workspace_d, sms,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int32_t tv_accept_noalloc(const uint16_t *logits_d, int32_t V, const int32_t *draft_tokens_d, const int32_t *parent_d,
                          const uint32_t *mask_d, int32_t B, int32_t nb, int32_t *argmax_d, int32_t *n_acc_d,
                          int32_t *path_d, int32_t *bonus_d, int32_t *dev_status_d, void *stream)
{
    if (nb < 0 || V < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)nb * B > TV_ACCEPT_NOALLOC_MAX_ROWS) return TV_ERR_UNSUPPORTED_SHAPE;
    if (!accept_shape_ok(V, B, nb)) return TV_ERR_UNSUPPORTED_SHAPE;
    if (!logits_d || !draft_tokens_d || !parent_d || !argmax_d || !n_acc_d || !path_d || !bonus_d)
        return TV_ERR_INVALID_ARG;
    if (!aligned(logits_d, 2) || !aligned(draft_tokens_d, 4) || !aligned(parent_d, 4) || !aligned(mask_d, 4) ||
        !aligned(argmax_d, 4) || !aligned(n_acc_d, 4) || !aligned(path_d, 4) || !aligned(bonus_d, 4) ||
        !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (nb == 0) return TV_OK;
    const int sms = sm_count();
    if (sms < 1) return TV_ERR_CUDA;
    cudaError_t e = tv::launch_accept_noalloc(logits_d, V, draft_tokens_d, parent_d, mask_d, B, nb, argmax_d, n_acc_d,
                                              path_d, bonus_d, dev_status_d, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int32_t tv_build_tree(const float *logp_d, const int32_t *tokens_d, int32_t nb, int32_t Dmax, int32_t K, int32_t B,
                      int32_t w, int32_t *parent_d, int32_t *token_d, float *score_d, int32_t *dev_status_d,
                      void *stream)
{
    if (nb < 0 || Dmax < 1 || K < 1 || w < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB || K > 32767 || Dmax > 32767) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)nb * Dmax * K >= (1ll << 31)) return TV_ERR_UNSUPPORTED_SHAPE;
    {  // the full tree of depth Dmax must hold B nodes
        long long total = 1, level = 1;
        for (int d = 1; d <= Dmax && total < B; ++d) {
            level *= K;
            total += level;
            if (level > B) level = B;
        }
        if (total < B) return TV_ERR_INVALID_ARG;
    }
    if (!logp_d || !tokens_d || !parent_d || !token_d || !score_d) return TV_ERR_INVALID_ARG;
    if (!aligned(logp_d, 4) || !aligned(tokens_d, 4) || !aligned(parent_d, 4) || !aligned(token_d, 4) ||
        !aligned(score_d, 4) || !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (nb == 0) return TV_OK;
    cudaError_t e = tv::launch_build_tree(logp_d, tokens_d, nb, Dmax, K, B, w, parent_d, token_d, score_d,
                                          dev_status_d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

size_t tv_gdn_tree_workspace_size(int32_t nb, int32_t B, int32_t H, int32_t D)
{
    if (nb < 0 || B < 1 || B > kMaxB || H < 1 || D != kHeadDim) return 0;
    return tv::gdn_workspace_bytes(nb, B, H);
}

int32_t tv_gdn_tree(const uint16_t *q_d, const uint16_t *k_d, const uint16_t *v_d, const float *alpha_d,
                    const float *beta_d, const float *S0_d, const int32_t *parent_d, int32_t nb, int32_t B, int32_t H,
                    int32_t D, float *O_d, void *workspace_d, size_t workspace_bytes, int32_t *dev_status_d,
                    void *stream)
{
    if (nb < 0 || H < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB || D != kHeadDim) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)nb * B * H * D >= (1ll << 31) || H > 65535 || nb > 65535) return TV_ERR_UNSUPPORTED_SHAPE;
    if (nb == 0) return TV_OK;
    if (!q_d || !k_d || !v_d || !alpha_d || !beta_d || !S0_d || !parent_d || !O_d) return TV_ERR_INVALID_ARG;
    if (!aligned(q_d, 16) || !aligned(k_d, 16) || !aligned(v_d, 16) || !aligned(S0_d, 16) || !aligned(O_d, 16) ||
        !aligned(alpha_d, 4) || !aligned(beta_d, 4) || !aligned(parent_d, 4) || !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (!workspace_d || !aligned(workspace_d, 16) || workspace_bytes < tv::gdn_workspace_bytes(nb, B, H))
        return TV_ERR_INVALID_ARG;
    cudaError_t e = tv::launch_gdn_tree(q_d, k_d, v_d, alpha_d, beta_d, S0_d, parent_d, nb, B, H, O_d, workspace_d,
                                        dev_status_d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int32_t tv_gdn_commit(const uint16_t *k_d, const uint16_t *v_d, const float *alpha_d, const float *beta_d,
                      const float *S0_d, const int32_t *n_acc_d, const int32_t *path_d, int32_t nb, int32_t B,
                      int32_t H, int32_t D, float *S_out_d, int32_t *dev_status_d, void *stream)
{
    if (nb < 0 || H < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB || D != kHeadDim) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)nb * B * H * D >= (1ll << 31) || H > 65535 || nb > 65535) return TV_ERR_UNSUPPORTED_SHAPE;
    if (nb == 0) return TV_OK;
    if (!k_d || !v_d || !alpha_d || !beta_d || !S0_d || !n_acc_d || !path_d || !S_out_d) return TV_ERR_INVALID_ARG;
    if (!aligned(k_d, 16) || !aligned(v_d, 16) || !aligned(S0_d, 4) || !aligned(S_out_d, 4) || !aligned(alpha_d, 4) ||
        !aligned(beta_d, 4) || !aligned(n_acc_d, 4) || !aligned(path_d, 4) || !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    cudaError_t e = tv::launch_gdn_commit(k_d, v_d, alpha_d, beta_d, S0_d, n_acc_d, path_d, nb, B, H, S_out_d,
                                          dev_status_d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int32_t tv_kv_commit(void *k_cache_d, void *v_cache_d, const int32_t *block_table_d, const int32_t *prefix_lens_d,
                     const int32_t *n_acc_d, const int32_t *path_d, int32_t nb, int32_t B, int32_t Hkv, int32_t D,
                     int32_t page_size, int32_t num_blocks, int32_t max_pages, int32_t *new_prefix_lens_d,
                     int32_t *dev_status_d, void *stream)
{
    if (nb < 0 || Hkv < 1 || num_blocks < 1 || max_pages < 1) return TV_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB || D != kHeadDim || page_size != kPageSize) return TV_ERR_UNSUPPORTED_SHAPE;
    if ((long long)nb * Hkv >= (1ll << 31) || (long long)num_blocks * Hkv * kPageSize >= (1ll << 31))
        return TV_ERR_UNSUPPORTED_SHAPE;
    if (!k_cache_d || !v_cache_d || !block_table_d || !prefix_lens_d || !n_acc_d || !path_d || !new_prefix_lens_d)
        return TV_ERR_INVALID_ARG;
    if (new_prefix_lens_d == prefix_lens_d) return TV_ERR_INVALID_ARG;
    if (!aligned(k_cache_d, 16) || !aligned(v_cache_d, 16) || !aligned(block_table_d, 4) ||
        !aligned(prefix_lens_d, 4) || !aligned(n_acc_d, 4) || !aligned(path_d, 4) || !aligned(new_prefix_lens_d, 4) ||
        !aligned(dev_status_d, 4))
        return TV_ERR_INVALID_ARG;
    if (nb == 0) return TV_OK;
    cudaError_t e = tv::launch_kv_commit(static_cast<uint16_t *>(k_cache_d), static_cast<uint16_t *>(v_cache_d),
                                         block_table_d, prefix_lens_d, n_acc_d, path_d, nb, B, Hkv, D, num_blocks,
                                         max_pages, new_prefix_lens_d, dev_status_d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

int32_t tv_selftest_wait(uint32_t limit_us, int32_t *dev_status_d, void *stream)
{
    if (limit_us < 1 || limit_us > 1000000u || !dev_status_d || !aligned(dev_status_d, 4)) return TV_ERR_INVALID_ARG;
    cudaError_t e = tv::launch_selftest_wait((uint64_t)limit_us * 1000ull, dev_status_d,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // extern "C"
