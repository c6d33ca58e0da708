/*
 * libtreeverify — the verify step of tree speculative decoding on one GB300
 * (sm_103a): ancestor masks, tree-causal paged attention, vocab argmax and
 * greedy tree acceptance.
 *
 * Sources (page title, section):
 *   [JF-2]  JETFLOW technical summary, §2 "Arquitectura Central": tree-causal
 *           attention mask — a draft-tree node attends to the input prefix and
 *           to its ancestors in the tree, never to descendants or to unrelated
 *           sibling branches (per-branch factorisation
 *           q(pi(v)|x) = prod_{u in pi(v)} q(y_u | x, h, pi_<u)).
 *   [JF-3]  JETFLOW summary, §3 "Contribuciones Clave" item 3: verification
 *           runs as paged FlashAttention with the tree mask staged in.
 *   [TfM-P] DFlash-TfM summary, "Declaración del Problema" item 3: standard
 *           tree verification = one target pass with ancestor-restricted
 *           masking.
 *   [TfM-3] DFlash-TfM summary, §3 "Solución": the tree is topologically
 *           ordered (parents before children).
 *   [JF-2t] JETFLOW summary, §2 "Estrategia de Entrenamiento", tree
 *           construction: logits for every depth at once, cumulative draft
 *           log-probability as the branch score, best-first expansion to a budget.
 *   [TfM-2t] DFlash-TfM summary, §2 "Construcción de Árboles": the top w
 *           candidates of the heap are expanded together (ceil(B/w) rounds).
 *   [TfM-3g] DFlash-TfM summary, §3 "Verificación de Árboles sin Rollback": the
 *           Gated DeltaNet state update, the masked triangular solve
 *           (I + X) U = beta V over the topologically ordered tree, and the state
 *           committed only once the accepted branch is known.
 *   [JF-4]  JETFLOW summary, §3 item 2 and §4: accepted tokens (tau) and
 *           longer accepted prefixes; the pages give no acceptance rule, so
 *           the greedy rule below is this library's reading.
 *
 * Conventions for every entry point
 *   - All pointers with a _d meaning are DEVICE pointers on the current
 *     device; the caller allocates and owns every buffer (workspaces
 *     included).  The library allocates no device memory, keeps no pointer
 *     after a call returns and encodes TMA descriptors on every call; its only
 *     host state is per-device: the SM count, the attention kernel's
 *     shared-memory opt-in and the device address of tv_accept_noalloc's
 *     scratch array.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on `stream` and returns; results
 *     are ready when the stream reaches that point.
 *   - Host-detectable problems (null pointers, sizes, alignment, unsupported
 *     shapes, workspace too small) are returned synchronously as a tv_status
 *     and nothing is enqueued.  Data-dependent problems found on the device
 *     (bad parent array, prefix too long for the block table, block id out of
 *     range, an internal wait that ran out) are written to *dev_status_d (a
 *     device int32 the caller zeroes beforehand; the first error code wins)
 *     and the affected outputs are unspecified.  Kernels never trap.
 *   - bf16 tensors are passed as raw 16-bit patterns.
 *   - Shape limits: 1 <= B <= 256, head dim D = 128, page size 16,
 *     Hq/Hkv = G in {1,2,4,8,16}.  Anything else returns
 *     TV_ERR_UNSUPPORTED_SHAPE; there is no fallback path.
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TV_API __attribute__((visibility("default")))
#else
#define TV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tv_status {
    TV_OK = 0,
    TV_ERR_INVALID_ARG = 1,       /* null pointer, bad size, misalignment, bad block id / prefix */
    TV_ERR_NOT_TOPOLOGICAL = 2,   /* parent[0] != -1 or parent[i] not in [0, i) */
    TV_ERR_UNSUPPORTED_SHAPE = 3, /* outside the supported shape set above */
    TV_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
    TV_ERR_TIMEOUT = 5,           /* a bounded device-side wait ran out (device status only) */
    TV_ERR_UNIMPLEMENTED = 6
} tv_status;

/* Human-readable name of a status code (static storage). */
TV_API const char *tv_status_str(int32_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
TV_API int32_t tv_version(void);

/*
 * Ancestor masks  [JF-2], [TfM-P], [TfM-3]
 *
 *   mask[b][i][w] bit j (j = 32*w + bit, LSB first) is 1 iff node j is node i
 *   or one of its ancestors:  anc[0] = {0},  anc[i] = anc[parent[i]] U {i}.
 *   depth[b][i] = number of edges from the root to node i.
 *
 *   parent_d  int32 [nb][B]    parent[b][0] = -1, 0 <= parent[b][i] < i
 *   mask_d    uint32 [nb][B][W], W = ceil(B/32)   (out; bits >= B are 0)
 *   depth_d   int32 [nb][B]    (out, may be NULL)
 *   dev_status_d  int32 device word (may be NULL); TV_ERR_NOT_TOPOLOGICAL is
 *                 written there when a parent array is invalid
 * Returns TV_OK, TV_ERR_INVALID_ARG (null mask/parent, nb < 0),
 * TV_ERR_UNSUPPORTED_SHAPE (B outside [1,256]) or TV_ERR_CUDA.
 */
TV_API int32_t tv_build_mask(const int32_t *parent_d, int32_t B, int32_t nb, uint32_t *mask_d,
                      int32_t *depth_d, int32_t *dev_status_d, void *stream);

/*
 * Tree-causal paged attention with split-KV merge
 * [JF-2], [JF-3], [TfM-P]
 *
 * For every sequence b, node i, query head h (kv head g = h / G):
 *   keys  j in [0, P_b)  U  { P_b + t : t in anc[i] }
 *   s_j   = scale * <q[b,i,h], K[b,g,j]>
 *   O     = sum_j softmax(s)_j V[b,g,j]       (bf16 out, fp32 accumulation)
 *   LSE   = ln sum_j exp(s_j)                  (fp32 out)
 * Logical position p of sequence b lives in physical page
 * block_table[b][p / 16], slot p % 16.  The caller has already written the
 * tree nodes' K/V at positions [P_b, P_b + B) (node t at P_b + t) and applied
 * RoPE (position P_b + depth[i] is the natural choice; tv_build_mask returns
 * depth).  Cache slots past P_b + B inside the last page must hold finite
 * values (zero-initialised caches satisfy this): they are multiplied by zero
 * probabilities.
 *
 * Value range: a row tile whose key range is split between CTAs parks its
 * normalised partial output in fp16 before the merge, so every V entry must
 * satisfy |v| <= 65504 (fp16's largest finite value; the partial output of a
 * row is a convex combination of V rows).  Larger values make only the split
 * rows overflow.  Activations of the models these shapes come from stay far
 * below that.
 */
typedef struct tv_attn_args {
    const void *q_d;             /* bf16 [nb*B][Hq][D], 16-byte aligned */
    const void *k_cache_d;       /* bf16 [num_blocks][Hkv][page_size][D], 16-byte aligned */
    const void *v_cache_d;       /* same layout as k_cache_d */
    const int32_t *block_table_d;/* int32 [nb][max_pages]; must cover P_b + B positions */
    const int32_t *prefix_lens_d;/* int32 [nb], P_b >= 0 (committed prefix, tree excluded) */
    const uint32_t *mask_d;      /* uint32 [nb][B][ceil(B/32)] from tv_build_mask, or NULL */
    void *o_d;                   /* bf16 [nb*B][Hq][D] (out), 16-byte aligned */
    float *lse_d;                /* fp32 [nb*B][Hq] (out), natural log */
    int32_t *dev_status_d;       /* device status word, may be NULL */
    int32_t nb, B, Hq, Hkv, D, page_size, num_blocks, max_pages;
    float scale;                 /* <= 0 selects 1/sqrt(D) */
    int32_t num_ctas;            /* 0 = one CTA per SM; otherwise the CTA count to use */
    const int32_t *parent_d;     /* int32 [nb][B], read only when mask_d is NULL: then each query
                                    row's ancestor bits come from a walk up its node's root path
                                    (the mask build folded into the attention; a parent array
                                    that is not topological writes TV_ERR_NOT_TOPOLOGICAL) */
} tv_attn_args;

/* Bytes of device workspace tv_attn needs for these arguments (depends on
 * num_ctas and the device's SM count; 0 never happens).  Returns 0 when the
 * arguments are invalid. */
TV_API size_t tv_attn_workspace_size(const tv_attn_args *args);

/* Enqueue the attention: one or two kernel launches on `stream`
 * (tv_attn_launches says which).  Row tiles whose key range is split between
 * CTAs leave normalised partial outputs (fp16) and LSEs (fp32) in the
 * workspace.  The CTAs form groups of NP = ceil(MT / 2) (MT = ceil(B / (128 /
 * (Hq / Hkv))) row tiles per (sequence, kv head) unit); with fewer groups than
 * twice the units (a split tile then has about two parts) the CTA whose part
 * of a tile lands last merges it, otherwise a second kernel merges every split
 * tile.  A small launch (every unit fits the CTA count at once and the block
 * table covers at most 8 KV tiles of 128 keys per sequence) gives each unit
 * its own CTAs and splits nothing.
 * workspace_d: device buffer of at least tv_attn_workspace_size(args) bytes,
 * 16-byte aligned.  It must be zero-filled (cudaMemset) before its first call;
 * besides the partials it holds arrival counters, at offsets that do not
 * depend on the arguments, which every call leaves zero, so a workspace can
 * serve calls of any shape after that.  A call whose dev_status_d reports
 * TV_ERR_TIMEOUT may leave counters behind: zero the workspace again before
 * reusing it.
 * Concurrent calls need separate workspaces.
 *
 * Ordering: the attention kernel is launched as a programmatic dependent of the
 * previous kernel on the stream and reads q, the caches, block_table and
 * prefix_lens before waiting for that kernel to finish (it waits only before
 * reading mask_d or parent_d).  So that previous kernel must not be one that writes those
 * inputs after signalling its dependents early.  Kernels launched without
 * programmatic dependent launch never signal early, and tv_build_mask (the
 * natural predecessor) writes only the masks and depths.
 *
 * Returns TV_OK, TV_ERR_INVALID_ARG, TV_ERR_UNSUPPORTED_SHAPE or TV_ERR_CUDA.
 * nb == 0 is a no-op. */
TV_API int32_t tv_attn(const tv_attn_args *args, void *workspace_d, size_t workspace_bytes, void *stream);

/* Kernel launches tv_attn enqueues for these arguments: 1 (the attention,
 * merging split tiles itself) or 2 (the attention, then the merge kernel);
 * 0 when nb == 0 or the arguments are invalid.  With num_ctas == 0 it asks the
 * current device for its SM count. */
TV_API int32_t tv_attn_launches(const tv_attn_args *args);

/*
 * Vocab argmax and greedy acceptance  [JF-4] (rule: this library's reading)
 *
 *   argmax[b*B+i] = first index of the maximum of logits[b*B+i][0..V)
 *                   (values compared as numbers, -0 == +0; a NaN counts as the maximum)
 *   ok[i]  = draft_tokens[b][i] == argmax[b*B + parent[b][i]]      (i >= 1)
 *   acc[i] = ok[j] for every j in anc[i] \ {0}                        (node 0 always accepted)
 *   v*     = the accepted node of greatest depth, smallest index on ties
 *   n_acc[b]   = depth[v*]  (accepted draft tokens, root excluded)
 *   path[b][k] = k-th node on the root-to-v* path (path[b][0] = 0), -1 after n_acc
 *   bonus[b]   = argmax[b*B + v*]  (the target's next token after the accepted path)
 *
 *   logits_d       bf16 [nb*B][V], 2-byte aligned (any V >= 1)
 *   draft_tokens_d int32 [nb][B]  (entry 0 of each sequence is ignored)
 *   parent_d       int32 [nb][B]  (the array given to tv_build_mask)
 *   mask_d         uint32 [nb][B][ceil(B/32)] from tv_build_mask for the same parent,
 *                  or NULL: the walk then builds each node's ancestor bits from
 *                  parent_d itself while the argmax runs (tv_build_mask is not
 *                  needed); a parent array that is not topological then writes
 *                  TV_ERR_NOT_TOPOLOGICAL and gives n_acc = 0, path = {0, -1, ...},
 *                  bonus = argmax of the root
 *   argmax_d       int32 [nb*B] (out), n_acc_d int32 [nb], path_d int32 [nb][B],
 *   bonus_d        int32 [nb] (out)
 *   workspace_d    device buffer of at least tv_accept_workspace_size(V, B, nb)
 *                  bytes (one 8-byte argmax key per logits row), 8-byte aligned,
 *                  ZEROED before the first call that uses it (cudaMemsetAsync
 *                  once): the argmax combines partial maxima into the keys with
 *                  atomic maxima, and the acceptance kernel sets every key it
 *                  reads back to zero, so each call leaves the workspace zeroed for
 *                  the next.  A call that returns TV_ERR_CUDA may leave keys behind:
 *                  zero the workspace again before reusing it.  Concurrent calls need
 *                  separate workspaces.
 * Returns TV_OK, TV_ERR_INVALID_ARG, TV_ERR_UNSUPPORTED_SHAPE (B outside
 * [1, 256], V > INT32_MAX - 8192, or nb * B * ceil(V / 4096) >= 2^31) or
 * TV_ERR_CUDA.  A parent array that is not topological is reported through
 * dev_status_d.
 */
TV_API size_t tv_accept_workspace_size(int32_t V, int32_t B, int32_t nb);

TV_API int32_t tv_accept(const uint16_t *logits_d, int32_t V, const int32_t *draft_tokens_d,
                         const int32_t *parent_d, const uint32_t *mask_d, int32_t B, int32_t nb,
                         int32_t *argmax_d, int32_t *n_acc_d, int32_t *path_d, int32_t *bonus_d,
                         int32_t *dev_status_d, void *workspace_d, size_t workspace_bytes, void *stream);

/*
 * Best-first draft-tree construction with top-w rounds  [JF-2t] [TfM-2t]
 *
 *   Per sequence: depth d (1..Dmax) offers K candidates, token tokens[b][d-1][c]
 *   with draft log-probability logp[b][d-1][c], sorted best first (c = 0 best);
 *   the same candidates hang under every node at depth d-1 (the draft head emits
 *   logits for every depth at once).  A candidate child (u, c) at depth d scores
 *   score[u] + logp[d-1][c] (fp32, cumulative draft log-probability); node 0 is
 *   the root (score 0).  Each round takes the min(w, B - made) best candidates
 *   (larger score, then smaller parent index, then smaller rank), numbers them in
 *   that order (so the tree is topologically ordered) and only then adds their
 *   children; w = 1 is plain best-first expansion, B nodes take ceil(B/w)
 *   rounds once the heap holds w candidates.
 *
 *   logp_d    fp32 [nb][Dmax][K], finite, non-increasing along c
 *   tokens_d  int32 [nb][Dmax][K]
 *   parent_d  int32 [nb][B] (out): -1 for the root; feeds tv_build_mask / tv_accept
 *   token_d   int32 [nb][B] (out): the draft token of each node, -1 for the root
 *   score_d   fp32 [nb][B] (out): cumulative log-probability, 0 for the root
 *   Limits: 1 <= B <= 256, 1 <= K <= 32767, 1 <= Dmax <= 32767, w >= 1, and the
 *   full tree of depth Dmax must hold B nodes (else TV_ERR_INVALID_ARG).
 * Ordering: a programmatic dependent of the previous kernel; waits for it before
 * reading anything.  Log-probs that are not finite or not sorted write
 * TV_ERR_INVALID_ARG to dev_status_d (outputs unspecified).
 */
TV_API int32_t tv_build_tree(const float *logp_d, const int32_t *tokens_d, int32_t nb, int32_t Dmax, int32_t K,
                             int32_t B, int32_t w, int32_t *parent_d, int32_t *token_d, float *score_d,
                             int32_t *dev_status_d, void *stream);

/*
 * Rollback-free tree verification through a Gated DeltaNet layer  [TfM-3g]
 *
 *   Per sequence b and head h, with the committed state S0[b][h] (D x D: rows
 *   indexed by the key dimension, columns by the value dimension), every tree
 *   node i gets the output of the state its own root path builds, without
 *   touching S0:
 *     S_i = alpha_i (I - beta_i k_i k_i^T) S_parent(i) + beta_i k_i v_i^T
 *     (S_parent(root) = S0),      o_i = S_i^T q_i.
 *   Computed as the masked triangular solve over the tree: with gamma_i the
 *   product of alpha on i's root path, (I + X) U = beta (V - gamma K S0) with
 *   X_ij = beta_i (gamma_i/gamma_j) k_i.k_j for j a strict ancestor of i, and
 *   O = gamma Q S0 + Y U with Y_ij = (gamma_i/gamma_j) q_i.k_j for j an ancestor
 *   of i or i itself.
 *
 *   q_d, k_d, v_d   bf16 [nb*B][H][D], 16-byte aligned (GDN layers normalise q, k)
 *   alpha_d, beta_d fp32 [nb*B][H]
 *   S0_d            fp32 [nb][H][D][D], 16-byte aligned
 *   parent_d        int32 [nb][B], topologically ordered (as tv_build_mask takes it)
 *   O_d             fp32 [nb*B][H][D] (out), 16-byte aligned
 *   workspace_d     >= tv_gdn_tree_workspace_size(nb, B, H, D) bytes, 16-byte
 *                   aligned: per (sequence, head, 32-column value slice) a B x B
 *                   table of 16-byte ancestor records, plus (B > 128) two fp32
 *                   [B][32] row blocks; concurrent calls need their own
 *   Shapes: D = 128, 1 <= B <= 256.
 * One kernel launch per call (4 CTAs per (sequence, head), one per 32 value
 * columns; tensor cores form the Gram blocks and the slice's K S0 and Q S0), a
 * programmatic dependent of the previous kernel
 * on the stream (it waits for it before reading anything).  A parent array that is
 * not topological writes TV_ERR_NOT_TOPOLOGICAL to dev_status_d (outputs
 * unspecified); an internal wait that runs out writes TV_ERR_TIMEOUT.
 * Returns TV_OK (nb == 0 launches nothing), TV_ERR_INVALID_ARG (null or misaligned
 * pointer, nb or H < 1, workspace too small), TV_ERR_UNSUPPORTED_SHAPE or TV_ERR_CUDA.
 * tv_gdn_tree_workspace_size returns 0 for an unsupported shape.
 */
TV_API size_t tv_gdn_tree_workspace_size(int32_t nb, int32_t B, int32_t H, int32_t D);
TV_API int32_t tv_gdn_tree(const uint16_t *q_d, const uint16_t *k_d, const uint16_t *v_d, const float *alpha_d,
                           const float *beta_d, const float *S0_d, const int32_t *parent_d, int32_t nb, int32_t B,
                           int32_t H, int32_t D, float *O_d, void *workspace_d, size_t workspace_bytes,
                           int32_t *dev_status_d, void *stream);

/*
 * Commit of a Gated DeltaNet layer's state for the accepted branch  [TfM-3g]
 *
 *   Tree verification (tv_gdn_tree) leaves the committed state S0 untouched; once
 *   the accepted branch is known the state is committed by applying the
 *   recurrence S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T from
 *   S0 to the nodes path[b][0] (the root) .. path[b][n_acc[b]], in that order.
 *   k_d, v_d        bf16 [nb*B][H][D] (the tree's tokens, as given to tv_gdn_tree), 16-byte aligned
 *   alpha_d, beta_d fp32 [nb*B][H]
 *   S0_d            fp32 [nb][H][D][D] (rows: key dimension)
 *   n_acc_d, path_d int32 [nb] and [nb][B] as tv_accept returns them
 *   S_out_d         fp32 [nb][H][D][D] (out); may be S0_d (committed in place)
 *   Shapes: D = 128, 1 <= B <= 256.
 * One kernel launch (8 CTAs per (sequence, head), one per 16 state columns), a
 * programmatic dependent of the previous kernel on the stream; it waits for it
 * before reading anything, so it may directly follow tv_accept.  A path that is not a root path of at most B
 * nodes (root first, strictly increasing, 0 <= n_acc < B) writes
 * TV_ERR_INVALID_ARG to dev_status_d and copies S0 to S_out unchanged.
 * Returns TV_OK (nb == 0 launches nothing), TV_ERR_INVALID_ARG, TV_ERR_UNSUPPORTED_SHAPE
 * or TV_ERR_CUDA.
 */
TV_API int32_t tv_gdn_commit(const uint16_t *k_d, const uint16_t *v_d, const float *alpha_d, const float *beta_d,
                             const float *S0_d, const int32_t *n_acc_d, const int32_t *path_d, int32_t nb,
                             int32_t B, int32_t H, int32_t D, float *S_out_d, int32_t *dev_status_d, void *stream);

/*
 * Commit of the accepted branch  [TfM-3] (the pages commit state once the
 * accepted branch is known; for a paged K/V cache this library reads that as
 * compaction in path order)
 *
 *   For sequence b with committed length P = prefix_lens[b] (tree node t at
 *   position P + t, as tv_attn reads it): position P + k of both caches takes
 *   what position P + path[b][k] held, for k = 1 .. n_acc[b] (the root stays at
 *   P; all rows are read before any is written), and
 *   new_prefix_lens[b] = P + n_acc[b] + 1.  No other position changes.
 *
 *   k_cache_d, v_cache_d   bf16 [num_blocks][Hkv][page_size][D] (in/out), 16-byte aligned
 *   block_table_d          int32 [nb][max_pages]; must cover P + B positions
 *   prefix_lens_d          int32 [nb]
 *   n_acc_d, path_d        int32 [nb] and [nb][B] as tv_accept returns them
 *   new_prefix_lens_d      int32 [nb] (out); must not be prefix_lens_d
 *   Shapes as tv_attn: 1 <= B <= 256, D = 128, page_size = 16.
 * Ordering: launched as a programmatic dependent of the previous kernel on the
 * stream, it waits for that kernel to finish before reading anything, so it can
 * directly follow tv_accept.
 * Returns TV_OK, TV_ERR_INVALID_ARG, TV_ERR_UNSUPPORTED_SHAPE or TV_ERR_CUDA.
 * A path that is not a root path of at most B nodes, an n_acc outside [0, B) or a
 * touched position the block table does not cover writes TV_ERR_INVALID_ARG to
 * dev_status_d and leaves that sequence uncommitted (new_prefix_lens_d[b] = P).
 */
TV_API int32_t tv_kv_commit(void *k_cache_d, void *v_cache_d, const int32_t *block_table_d,
                            const int32_t *prefix_lens_d, const int32_t *n_acc_d, const int32_t *path_d,
                            int32_t nb, int32_t B, int32_t Hkv, int32_t D, int32_t page_size, int32_t num_blocks,
                            int32_t max_pages, int32_t *new_prefix_lens_d, int32_t *dev_status_d, void *stream);

/*
 * Argmax and acceptance in one kernel  [JF-4]
 *
 * The same results as tv_accept (argmax of every row, then the greedy walk), from
 * one kernel launch instead of two: the argmax CTAs own whole rows, and the CTA
 * whose keys complete a sequence's B rows (a per-sequence counter in the
 * workspace tells) runs that sequence's walk.
 *   mask_d     as tv_accept, or NULL: then the walk builds each node's ancestor
 *              bits from parent_d itself (tv_build_mask is not needed), and a
 *              parent array that is not topological writes TV_ERR_NOT_TOPOLOGICAL
 *              and gives n_acc = 0, path = {0, -1, ...}, bonus = argmax of the root
 *   workspace_d >= tv_accept_fused_workspace_size(V, B, nb) bytes, 8-byte aligned:
 *              nb*B 8-byte keys, then nb 32-bit counters.  The counters must be zero
 *              before the first call on a workspace (cudaMemset once); every call
 *              leaves them zero.  Concurrent calls need their own workspace.
 *   Other arguments as tv_accept.
 * Ordering: a programmatic dependent of the previous kernel on the stream; it
 * waits for it before reading anything.
 * Returns TV_OK, TV_ERR_INVALID_ARG, TV_ERR_UNSUPPORTED_SHAPE or TV_ERR_CUDA.
 */
TV_API size_t tv_accept_fused_workspace_size(int32_t V, int32_t B, int32_t nb);
TV_API int32_t tv_accept_fused(const uint16_t *logits_d, int32_t V, const int32_t *draft_tokens_d,
                               const int32_t *parent_d, const uint32_t *mask_d, int32_t B, int32_t nb,
                               int32_t *argmax_d, int32_t *n_acc_d, int32_t *path_d, int32_t *bonus_d,
                               int32_t *dev_status_d, void *workspace_d, size_t workspace_bytes, void *stream);

/*
 * tv_accept_noalloc — tv_accept for callers that cannot allocate device memory.
 * (The pages have no counterpart: this is an integration aid, not part of the
 * method.)
 *
 * Some callers cannot call cudaMalloc, and so cannot hand tv_accept a workspace:
 * code that runs while a stream is being captured into a CUDA graph (an
 * allocation there is not part of the graph and breaks the capture), and
 * serving runtimes that plan every device buffer at start-up and forbid
 * allocation on the decode path.  This entry point takes the same arguments as
 * tv_accept minus the workspace and computes the same results, with its scratch
 * (8 bytes per logits row, 64 KB in all) in a fixed array inside the library
 * image.
 *
 *   - Limit: nb * B <= TV_ACCEPT_NOALLOC_MAX_ROWS; larger calls return
 *     TV_ERR_UNSUPPORTED_SHAPE and enqueue nothing, as do V > INT32_MAX - 8192
 *     and the other shape limits of tv_accept.
 *   - The array exists once per GPU that loads the library and stays allocated
 *     until the process exits.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it together with the id of the device's
 *     context; make that first call before any stream capture.  After
 *     cudaDeviceReset the next call sees a new context and looks the address
 *     up again (the module, and so the array, may move), so make that call
 *     outside a capture too.
 *   - Every call on a device shares the array.  The array starts at zero when the
 *     library is loaded and every call leaves it at zero (the argmax combines
 *     into it with atomic maxima, the acceptance kernel resets what it read); if
 *     a call returns TV_ERR_CUDA, the next call on that device first launches a
 *     small kernel that zeroes it again.  Calls whose work overlaps on the GPU
 *     (different streams, no ordering between them) race on the array and their
 *     results are undefined: order them on one stream.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define TV_ACCEPT_NOALLOC_MAX_ROWS 8192
TV_API int32_t tv_accept_noalloc(const uint16_t *logits_d, int32_t V, const int32_t *draft_tokens_d,
                                 const int32_t *parent_d, const uint32_t *mask_d, int32_t B, int32_t nb,
                                 int32_t *argmax_d, int32_t *n_acc_d, int32_t *path_d, int32_t *bonus_d,
                                 int32_t *dev_status_d, void *stream);

/*
 * tv_selftest_wait — exercises the failure path of the bounded device waits.
 * (The pages have no counterpart: this checks the library's own fault handling.)
 *
 * The pipelined kernels (tv_attn, tv_gdn_tree) wait on shared-memory barriers
 * with a time limit; a wait that runs out writes TV_ERR_TIMEOUT to
 * *dev_status_d, stops the kernel cleanly (copies in flight land, tensor memory
 * is freed) and leaves the context usable.  This call launches one small kernel
 * that allocates tensor memory, waits on a barrier that nothing arrives at for
 * limit_us microseconds, reports TV_ERR_TIMEOUT, frees the tensor memory and
 * returns, so a test can see that path work without breaking a real kernel.
 *
 *   limit_us      1 .. 1000000
 *   dev_status_d  device int32, required (the caller zeroes it first)
 * Returns TV_OK (kernel enqueued), TV_ERR_INVALID_ARG or TV_ERR_CUDA.
 */
TV_API int32_t tv_selftest_wait(uint32_t limit_us, int32_t *dev_status_d, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H */
