/*
 * Tree-verification oracle: a plain, slow, fp64 CPU statement of what one
 * verify step of tree speculative decoding computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA library (no headers, no tables, no helpers) and the library never calls
 * it.
 *
 * Sources (page title, section):
 *  - JETFLOW summary, §2 "Arquitectura Central", tree-causal attention mask:
 *    a draft-tree node attends to the original input prefix and to its
 *    ancestors inside the tree, never to its descendants or to unrelated
 *    sibling branches; this imposes the per-branch factorisation
 *    q(pi(v)|x) = prod_{u in pi(v)} q(y_u | x, h, pi_<u).
 *  - JETFLOW summary, §3 item 3: verification runs as paged attention with a
 *    tree mask (paged KV cache, block table).
 *  - DFlash-TfM summary, "Declaración del Problema" item 3: tree verification
 *    by ancestor-restricted attention masking; §3 "Solución": the tree is
 *    topologically ordered.
 *  - Acceptance: the pages speak of "accepted tokens" and "longer accepted
 *    prefixes" (JETFLOW §3 item 2, §4) without a rule.  The rule used here is
 *    greedy: a node is accepted when its parent is accepted and its draft token
 *    equals the target argmax at its parent; the deepest accepted node wins,
 *    ties going to the smallest node index.
 *
 * Readings taken where the pages are silent: a node attends to itself; tree
 * node t's K/V sit at logical position prefix_len + t of the paged cache;
 * query head h uses kv head h / (Hq/Hkv); scale defaults to 1/sqrt(D); LSE is
 * the natural log of sum(exp(scaled score)); the argmax is the first index of
 * the maximum, a NaN counting as the maximum.
 *
 * Every function returns 0 on success, 1 for a bad argument, 2 for a parent
 * array that is not a topologically ordered single-root tree.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define TVO_OK 0
#define TVO_ERR_ARG 1
#define TVO_ERR_NOT_TOPOLOGICAL 2

/* bf16 bit pattern -> double (exact: bf16 is the top half of an IEEE binary32). */
static double bf16_value(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* A parent array is valid when node 0 is the only root and every other node's
 * parent has a smaller index (DFlash-TfM summary, §3: topological order). */
static int parent_is_valid(const int32_t *parent, int B)
{
    if (parent[0] != -1) return 0;
    for (int i = 1; i < B; i++)
        if (parent[i] < 0 || parent[i] >= i) return 0;
    return 1;
}

/* anc[i*B + j] = 1 when node j lies on the root-to-i path (i itself included). */
static void ancestor_sets(const int32_t *parent, int B, uint8_t *anc)
{
    memset(anc, 0, (size_t)B * B);
    for (int i = 0; i < B; i++) {
        int j = i;
        while (j != -1) {
            anc[(size_t)i * B + j] = 1;
            j = parent[j];
        }
    }
}

/* ------------------------------------------------------------------ mask */

/* Packed ancestor masks: bit j of node i (word j/32, bit j%32, LSB first) is
 * set when node j is node i or one of its ancestors; depth[i] counts the edges
 * from the root to i.  mask: [nb][B][ceil(B/32)] words, depth: [nb][B]. */
int tvo_build_mask(const int32_t *parent, int B, int nb, uint32_t *mask, int32_t *depth)
{
    if (!parent || !mask || B < 1 || nb < 0) return TVO_ERR_ARG;
    const int W = (B + 31) / 32;
    for (int b = 0; b < nb; b++) {
        const int32_t *p = parent + (size_t)b * B;
        if (!parent_is_valid(p, B)) return TVO_ERR_NOT_TOPOLOGICAL;
        for (int i = 0; i < B; i++) {
            uint32_t *row = mask + ((size_t)b * B + i) * W;
            memset(row, 0, sizeof(uint32_t) * W);
            int j = i, d = 0;
            row[j / 32] |= 1u << (j % 32);
            while (p[j] != -1) {
                j = p[j];
                row[j / 32] |= 1u << (j % 32);
                d++;
            }
            if (depth) depth[(size_t)b * B + i] = d;
        }
    }
    return TVO_OK;
}

/* ------------------------------------------------------------- attention */

typedef struct {
    const uint16_t *q;          /* [nb*B][Hq][D] bf16 */
    const uint16_t *k_cache;    /* [num_blocks][Hkv][page][D] bf16 */
    const uint16_t *v_cache;
    const int32_t *block_table; /* [nb][max_pages] */
    const int32_t *prefix_lens; /* [nb] */
    const int32_t *parent;      /* [nb][B] */
    int nb, B, Hq, Hkv, D, page, max_pages, num_blocks;
    double scale;
    long key_lo, key_hi;        /* only logical positions in [key_lo, key_hi) take part */
    double *O;                  /* [nb*B][Hq][D] */
    double *LSE;                /* [nb*B][Hq] */
    /* work distribution */
    long next_task;
    int error;
} attn_job;

/* Tree-causal attention for one (sequence b, query head h), every node. */
static int attn_one(attn_job *a, int b, int h)
{
    const int B = a->B, D = a->D, G = a->Hq / a->Hkv, g = h / G;
    const long P = a->prefix_lens[b];
    uint8_t *anc = malloc((size_t)B * B);
    long *pos = malloc(sizeof(long) * (size_t)(P + B));
    double *s = malloc(sizeof(double) * (size_t)(P + B));
    double *acc = malloc(sizeof(double) * (size_t)D);
    int rc = TVO_OK;
    if (!anc || !pos || !s || !acc) { rc = TVO_ERR_ARG; goto done; }
    ancestor_sets(a->parent + (size_t)b * B, B, anc);

    for (int i = 0; i < B; i++) {
        /* The keys node i may see: the whole prefix, then its root path. */
        long n = 0;
        for (long j = 0; j < P; j++) pos[n++] = j;
        for (int t = 0; t < B; t++)
            if (anc[(size_t)i * B + t]) pos[n++] = P + t;
        /* Optional restriction to a key range (used for split-range checks). */
        long m = 0;
        for (long k = 0; k < n; k++)
            if (pos[k] >= a->key_lo && (a->key_hi < 0 || pos[k] < a->key_hi)) pos[m++] = pos[k];
        n = m;

        const uint16_t *qrow = a->q + (((size_t)b * B + i) * a->Hq + h) * D;
        double *orow = a->O + (((size_t)b * B + i) * a->Hq + h) * D;
        double *lse = a->LSE + ((size_t)b * B + i) * a->Hq + h;

        /* Scores s_k = scale * <q, k_k>, read through the block table. */
        double smax = -INFINITY;
        for (long k = 0; k < n; k++) {
            long page_id = a->block_table[(size_t)b * a->max_pages + pos[k] / a->page];
            long slot = pos[k] % a->page;
            if (page_id < 0 || page_id >= a->num_blocks) { rc = TVO_ERR_ARG; goto done; }
            const uint16_t *krow = a->k_cache + (((size_t)page_id * a->Hkv + g) * a->page + slot) * D;
            double dot = 0.0;
            for (int d = 0; d < D; d++) dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
            s[k] = a->scale * dot;
            if (s[k] > smax) smax = s[k];
        }
        if (n == 0) {
            for (int d = 0; d < D; d++) orow[d] = 0.0;
            *lse = -INFINITY;
            continue;
        }
        /* Softmax with the maximum subtracted, then the weighted sum of V rows. */
        double l = 0.0;
        for (int d = 0; d < D; d++) acc[d] = 0.0;
        for (long k = 0; k < n; k++) {
            double w = exp(s[k] - smax);
            l += w;
            long page_id = a->block_table[(size_t)b * a->max_pages + pos[k] / a->page];
            long slot = pos[k] % a->page;
            const uint16_t *vrow = a->v_cache + (((size_t)page_id * a->Hkv + g) * a->page + slot) * D;
            for (int d = 0; d < D; d++) acc[d] += w * bf16_value(vrow[d]);
        }
        for (int d = 0; d < D; d++) orow[d] = acc[d] / l;
        *lse = smax + log(l);
    }
done:
    free(anc); free(pos); free(s); free(acc);
    return rc;
}

static void *attn_worker(void *arg)
{
    attn_job *a = arg;
    const long ntasks = (long)a->nb * a->Hq;
    for (;;) {
        long t = __atomic_fetch_add(&a->next_task, 1, __ATOMIC_RELAXED);
        if (t >= ntasks) break;
        int rc = attn_one(a, (int)(t / a->Hq), (int)(t % a->Hq));
        if (rc) __atomic_store_n(&a->error, rc, __ATOMIC_RELAXED);
    }
    return NULL;
}

/* O[b*B+i][h][:] and LSE[b*B+i][h] for every node and query head.
 * scale <= 0 selects 1/sqrt(D).  key_hi < 0 means no upper limit.
 * nthreads <= 0 uses every online host core.  Returns the thread count used
 * through *threads_used when that pointer is not null. */
int tvo_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
             const int32_t *block_table, const int32_t *prefix_lens, const int32_t *parent,
             int nb, int B, int Hq, int Hkv, int D, int page, int max_pages, int num_blocks,
             double scale, long key_lo, long key_hi, double *O, double *LSE,
             int nthreads, int *threads_used)
{
    if (!q || !k_cache || !v_cache || !block_table || !prefix_lens || !parent || !O || !LSE)
        return TVO_ERR_ARG;
    if (nb < 0 || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || page < 1) return TVO_ERR_ARG;
    for (int b = 0; b < nb; b++) {
        if (!parent_is_valid(parent + (size_t)b * B, B)) return TVO_ERR_NOT_TOPOLOGICAL;
        long need = ((long)prefix_lens[b] + B + page - 1) / page;
        if (prefix_lens[b] < 0 || need > max_pages) return TVO_ERR_ARG;
    }
    attn_job a = {q, k_cache, v_cache, block_table, prefix_lens, parent,
                  nb, B, Hq, Hkv, D, page, max_pages, num_blocks,
                  scale > 0 ? scale : 1.0 / sqrt((double)D), key_lo, key_hi, O, LSE, 0, 0};
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if ((long)nthreads > (long)nb * Hq && nb * Hq > 0) nthreads = nb * Hq;
    pthread_t *tid = malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid) return TVO_ERR_ARG;
    for (int t = 0; t < nthreads; t++) pthread_create(&tid[t], NULL, attn_worker, &a);
    for (int t = 0; t < nthreads; t++) pthread_join(tid[t], NULL);
    free(tid);
    if (threads_used) *threads_used = nthreads;
    return a.error;
}

/* Combine attention results computed over disjoint key ranges:
 * lse = ln sum_u exp(lse_u), O = sum_u exp(lse_u - lse) O_u.
 * O_parts: [U][rows][D], lse_parts: [U][rows]. */
int tvo_lse_merge(int U, long rows, int D, const double *O_parts, const double *lse_parts,
                  double *O, double *lse)
{
    if (U < 1 || rows < 0 || D < 1 || !O_parts || !lse_parts || !O || !lse) return TVO_ERR_ARG;
    for (long r = 0; r < rows; r++) {
        double m = -INFINITY;
        for (int u = 0; u < U; u++)
            if (lse_parts[(size_t)u * rows + r] > m) m = lse_parts[(size_t)u * rows + r];
        double *orow = O + (size_t)r * D;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            for (int d = 0; d < D; d++) orow[d] = 0.0;
            continue;
        }
        double sum = 0.0;
        for (int u = 0; u < U; u++) sum += exp(lse_parts[(size_t)u * rows + r] - m);
        lse[r] = m + log(sum);
        for (int d = 0; d < D; d++) orow[d] = 0.0;
        for (int u = 0; u < U; u++) {
            double w = exp(lse_parts[(size_t)u * rows + r] - lse[r]);
            const double *part = O_parts + ((size_t)u * rows + r) * D;
            for (int d = 0; d < D; d++) orow[d] += w * part[d];
        }
    }
    return TVO_OK;
}

/* ---------------------------------------------------------------- argmax */

/* am[r] = the first index of the maximum of row r (bf16 values compared as
 * real numbers, so -0 == +0); the first NaN, if any, counts as the maximum. */
int tvo_argmax(const uint16_t *logits, long rows, long V, int32_t *am)
{
    if (!logits || !am || rows < 0 || V < 1) return TVO_ERR_ARG;
    for (long r = 0; r < rows; r++) {
        const uint16_t *row = logits + (size_t)r * V;
        long best = 0;
        double bv = bf16_value(row[0]);
        for (long v = 1; v < V && !isnan(bv); v++) {
            double x = bf16_value(row[v]);
            if (isnan(x) || x > bv) { best = v; bv = x; }
        }
        am[r] = (int32_t)best;
    }
    return TVO_OK;
}

/* ------------------------------------------------------------ acceptance */

/* Greedy tree acceptance for nb sequences of B nodes.
 *   argmax_out [nb*B]: target argmax at every node (tvo_argmax of its logits row)
 *   n_acc [nb]:        depth of the chosen node = accepted draft tokens (root excluded)
 *   path [nb][B]:      node indices from the root (path[0] = 0) to the chosen node, then -1
 *   bonus [nb]:        target argmax at the chosen node (the next committed token)
 * Node 0 is the root and is always accepted; draft[b][0] is not read. */
int tvo_accept(const uint16_t *logits, long V, const int32_t *draft, const int32_t *parent,
               int B, int nb, int32_t *argmax_out, int32_t *n_acc, int32_t *path, int32_t *bonus)
{
    if (!logits || !draft || !parent || !argmax_out || !n_acc || !path || !bonus) return TVO_ERR_ARG;
    if (B < 1 || nb < 0 || V < 1) return TVO_ERR_ARG;
    int *acc = malloc(sizeof(int) * (size_t)B);
    int *dep = malloc(sizeof(int) * (size_t)B);
    if (!acc || !dep) { free(acc); free(dep); return TVO_ERR_ARG; }
    int rc = TVO_OK;
    for (int b = 0; b < nb && rc == TVO_OK; b++) {
        const int32_t *p = parent + (size_t)b * B;
        const int32_t *dr = draft + (size_t)b * B;
        int32_t *am = argmax_out + (size_t)b * B;
        if (!parent_is_valid(p, B)) { rc = TVO_ERR_NOT_TOPOLOGICAL; break; }
        tvo_argmax(logits + (size_t)b * B * V, B, V, am);

        acc[0] = 1;
        dep[0] = 0;
        for (int i = 1; i < B; i++) {
            dep[i] = dep[p[i]] + 1;
            acc[i] = acc[p[i]] && dr[i] == am[p[i]];
        }
        int best = 0;
        for (int i = 1; i < B; i++)
            if (acc[i] && dep[i] > dep[best]) best = i;

        n_acc[b] = dep[best];
        bonus[b] = am[best];
        int32_t *pr = path + (size_t)b * B;
        for (int k = 0; k < B; k++) pr[k] = -1;
        for (int k = dep[best], j = best; k >= 0; k--, j = p[j]) pr[k] = j;
    }
    free(acc); free(dep);
    return rc;
}

/* ------------------------------------------------------------ KV commit */

/* Commit of the accepted branch (DFlash-TfM summary, §3 "Solución": the state is
 * committed once the accepted branch is known, so nothing is rolled back).  For
 * attention the state is the paged K/V cache.  Sequence b holds its committed
 * tokens at logical positions [0, P) (P = prefix_lens[b]) and tree node t at
 * P + t.  The commit keeps the root and the accepted nodes, in path order:
 * afterwards position P + k holds what position P + path[b][k] held before, for
 * k = 0 .. n_acc[b] (path[b][0] = 0, so the root stays), and the committed
 * length becomes P + n_acc[b] + 1.  No other position changes.  All sources are
 * read before any destination is written (a source may be another row's
 * destination).  Logical position x of sequence b lives in physical page
 * block_table[b][x / page], slot x % page; caches are [num_blocks][Hkv][page][D]. */
int tvo_kv_commit(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_table, const int32_t *prefix_lens,
                  const int32_t *n_acc, const int32_t *path, int nb, int B, int Hkv, int D, int page, int max_pages,
                  int num_blocks, int32_t *new_prefix_lens)
{
    if (!k_cache || !v_cache || !block_table || !prefix_lens || !n_acc || !path || !new_prefix_lens) return TVO_ERR_ARG;
    if (nb < 0 || B < 1 || Hkv < 1 || D < 1 || page < 1 || max_pages < 1 || num_blocks < 1) return TVO_ERR_ARG;
    const size_t row = (size_t)D;                 /* elements of one (position, kv head) row */
    uint16_t *tmp = malloc(sizeof(uint16_t) * 2 * (size_t)B * Hkv * row);
    if (!tmp) return TVO_ERR_ARG;
    int rc = TVO_OK;
    for (int b = 0; b < nb && rc == TVO_OK; b++) {
        const int P = prefix_lens[b], n = n_acc[b];
        const int32_t *pr = path + (size_t)b * B;
        const int32_t *bt = block_table + (size_t)b * max_pages;
        if (P < 0 || n < 0 || n >= B || pr[0] != 0) { rc = TVO_ERR_ARG; break; }
        for (int k = 1; k <= n; k++)
            if (pr[k] <= pr[k - 1] || pr[k] >= B) rc = TVO_ERR_ARG;
        if ((long)P + B > (long)max_pages * page) rc = TVO_ERR_ARG;
        if (rc != TVO_OK) break;
        /* read every source row first */
        for (int k = 0; k <= n; k++) {
            const long x = (long)P + pr[k];
            const int blk = bt[x / page];
            if (blk < 0 || blk >= num_blocks) { rc = TVO_ERR_ARG; break; }
            for (int g = 0; g < Hkv; g++) {
                const size_t src = (((size_t)blk * Hkv + g) * page + (size_t)(x % page)) * row;
                memcpy(tmp + ((size_t)(2 * k) * Hkv + g) * row, k_cache + src, sizeof(uint16_t) * row);
                memcpy(tmp + ((size_t)(2 * k + 1) * Hkv + g) * row, v_cache + src, sizeof(uint16_t) * row);
            }
        }
        if (rc != TVO_OK) break;
        /* then write position P + k */
        for (int k = 0; k <= n; k++) {
            const long x = (long)P + k;
            const int blk = bt[x / page];
            if (blk < 0 || blk >= num_blocks) { rc = TVO_ERR_ARG; break; }
            for (int g = 0; g < Hkv; g++) {
                const size_t dst = (((size_t)blk * Hkv + g) * page + (size_t)(x % page)) * row;
                memcpy(k_cache + dst, tmp + ((size_t)(2 * k) * Hkv + g) * row, sizeof(uint16_t) * row);
                memcpy(v_cache + dst, tmp + ((size_t)(2 * k + 1) * Hkv + g) * row, sizeof(uint16_t) * row);
            }
        }
        new_prefix_lens[b] = P + n + 1;
    }
    free(tmp);
    return rc;
}

/* ---------------------------------------------------------- tree building */

/* Best-first draft-tree construction with top-w rounds.
 * JETFLOW summary, §2 "Estrategia de Entrenamiento" / tree construction: the
 * draft head emits logits for every tree depth at once, a branch score (by
 * default the cumulative draft log-probability) ranks the nodes and best-first
 * expansion builds the tree up to a budget.  DFlash-TfM summary, §2
 * "Construcción de Árboles": the top w candidates are taken from the candidate
 * heap and expanded together, so B nodes take ceil(B/w) rounds.
 * Reading: depth d's candidates are the K tokens tok[d][c] with log-probs
 * logp[d][c] (c = 0..K-1, per sequence), the same for every node at depth d-1;
 * a candidate child (node u, rank c) at depth d scores score[u] + logp[d][c] in
 * fp32 (the rounding the GPU uses); node 0 is the root (score 0, depth 0).
 * Each round takes the w best candidates in the heap (larger score first; ties to
 * the smaller parent index, then the smaller rank), numbers them in that order
 * and only then pushes their K children (depth < Dmax).  Outputs per sequence:
 * parent[b][i] (-1 for the root), token[b][i] (-1 for the root), score[b][i].
 * logp/tok are [nb][Dmax][K] (depth d at index d-1). */
typedef struct { float s; int u, c; } tvo_cand;

static int cand_better(const tvo_cand *a, const tvo_cand *b)
{
    if (a->s != b->s) return a->s > b->s;
    if (a->u != b->u) return a->u < b->u;
    return a->c < b->c;
}

int tvo_build_tree(const float *logp, const int32_t *tok, int nb, int Dmax, int K, int B, int w, int32_t *parent,
                   int32_t *token, float *score)
{
    if (!logp || !tok || !parent || !token || !score || nb < 0 || Dmax < 1 || K < 1 || B < 1 || w < 1)
        return TVO_ERR_ARG;
    {   /* the full tree of depth Dmax must hold B nodes */
        long total = 1, level = 1;
        for (int d = 1; d <= Dmax && total < B; d++) { level *= K; total += level; if (level > B) level = B; }
        if (total < B) return TVO_ERR_ARG;
    }
    /* a plain array of candidates; each round scans it w times (slow and obvious) */
    const long cap = (long)B * K + 1;
    tvo_cand *pool = malloc(sizeof(tvo_cand) * (size_t)cap);
    int *dep = malloc(sizeof(int) * (size_t)B);
    tvo_cand *round_sel = malloc(sizeof(tvo_cand) * (size_t)w);
    if (!pool || !dep || !round_sel) { free(pool); free(dep); free(round_sel); return TVO_ERR_ARG; }
    for (int b = 0; b < nb; b++) {
        const float *lp = logp + (size_t)b * Dmax * K;
        const int32_t *tk = tok + (size_t)b * Dmax * K;
        int32_t *par = parent + (size_t)b * B, *tkn = token + (size_t)b * B;
        float *sc = score + (size_t)b * B;
        par[0] = -1; tkn[0] = -1; sc[0] = 0.f; dep[0] = 0;
        long np = 0;
        for (int c = 0; c < K; c++) { pool[np].s = 0.f + lp[c]; pool[np].u = 0; pool[np].c = c; np++; }
        int made = 1;
        while (made < B && np > 0) {
            int take = w < B - made ? w : B - made;
            int got = 0;
            for (int t = 0; t < take && np > 0; t++) {
                long best = 0;
                for (long j = 1; j < np; j++)
                    if (cand_better(&pool[j], &pool[best])) best = j;
                round_sel[got++] = pool[best];
                pool[best] = pool[--np];
            }
            int first = made;
            for (int t = 0; t < got; t++) {
                const int i = made++;
                par[i] = round_sel[t].u;
                dep[i] = dep[round_sel[t].u] + 1;
                tkn[i] = tk[(size_t)(dep[i] - 1) * K + round_sel[t].c];
                sc[i] = round_sel[t].s;
            }
            for (int i = first; i < made; i++)
                if (dep[i] < Dmax)
                    for (int c = 0; c < K; c++) {
                        pool[np].s = sc[i] + lp[(size_t)dep[i] * K + c];
                        pool[np].u = i; pool[np].c = c; np++;
                    }
        }
    }
    free(pool); free(dep); free(round_sel);
    return TVO_OK;
}

/* ------------------------------------------------- Gated DeltaNet over a tree */

/* Tree verification through a Gated DeltaNet layer (DFlash-TfM summary, §3
 * "Verificación de Árboles sin Rollback"): the recurrent state follows
 *   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 * (S is D x D: rows indexed by the key dimension, columns by the value
 * dimension), and every tree node must see the state its own root path would
 * have built from the committed state S0, without touching S0 (no rollback).
 * Reading: node i's state is the recurrence applied along root ... i starting
 * from S0 (parent[i] = -1 for the root, which is itself a tree node), and its
 * output is o_i = S_i^T q_i.  This is the plain definition, applied by brute force
 * per node and head, in fp64.
 *   q, k, v: bf16 [nb*B][H][D]; alpha, beta: fp32 [nb*B][H]; S0: fp32 [nb][H][D][D];
 *   parent: int32 [nb][B] topologically ordered; O: fp64 [nb*B][H][D]. */
int tvo_gdn_tree(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta,
                 const float *S0, const int32_t *parent, int nb, int B, int H, int D, double *O)
{
    if (!q || !k || !v || !alpha || !beta || !S0 || !parent || !O || nb < 0 || B < 1 || H < 1 || D < 1)
        return TVO_ERR_ARG;
    double *S = malloc(sizeof(double) * (size_t)D * D);
    double *kv = malloc(sizeof(double) * (size_t)D * 3);
    int *path = malloc(sizeof(int) * (size_t)B);
    if (!S || !kv || !path) { free(S); free(kv); free(path); return TVO_ERR_ARG; }
    int rc = TVO_OK;
    for (int b = 0; b < nb && rc == TVO_OK; b++) {
        const int32_t *p = parent + (size_t)b * B;
        if (!parent_is_valid(p, B)) { rc = TVO_ERR_NOT_TOPOLOGICAL; break; }
        for (int h = 0; h < H; h++) {
            for (int i = 0; i < B; i++) {
                int len = 0;
                for (int j = i; j != -1; j = p[j]) path[len++] = j;
                const float *s0 = S0 + ((size_t)b * H + h) * D * D;
                for (int x = 0; x < D * D; x++) S[x] = s0[x];
                for (int t = len - 1; t >= 0; t--) {          /* root first */
                    const size_t row = ((size_t)b * B + path[t]) * H + h;
                    const double a = alpha[row], be = beta[row];
                    double *kk = kv, *vv = kv + D, *ks = kv + 2 * D;
                    for (int d = 0; d < D; d++) { kk[d] = bf16_value(k[row * D + d]); vv[d] = bf16_value(v[row * D + d]); }
                    for (int c = 0; c < D; c++) {                /* ks = k^T S (one entry per value column) */
                        double acc = 0.0;
                        for (int r = 0; r < D; r++) acc += kk[r] * S[(size_t)r * D + c];
                        ks[c] = acc;
                    }
                    for (int r = 0; r < D; r++)
                        for (int c = 0; c < D; c++)
                            S[(size_t)r * D + c] = a * (S[(size_t)r * D + c] - be * kk[r] * ks[c]) + be * kk[r] * vv[c];
                }
                const size_t row = ((size_t)b * B + i) * H + h;
                for (int c = 0; c < D; c++) {
                    double acc = 0.0;
                    for (int r = 0; r < D; r++) acc += S[(size_t)r * D + c] * bf16_value(q[row * D + r]);
                    O[row * D + c] = acc;
                }
            }
        }
    }
    free(S); free(kv); free(path);
    return rc;
}

/* Commit of a Gated DeltaNet layer's state for the accepted branch (DFlash-TfM
 * summary, §3: the state is committed only in the next decoding iteration, once
 * the accepted branch is known, so nothing is rolled back).  Per sequence b and
 * head h the recurrence
 *   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 * is applied from S0 to the nodes path[b][0] (the root) .. path[b][n_acc[b]] in
 * that order, in fp64, and the result is the new committed state.  The path is
 * checked as tvo_kv_commit checks it (root first, strictly increasing, inside the
 * tree, 0 <= n_acc < B).
 *   k, v: bf16 [nb*B][H][D]; alpha, beta: fp32 [nb*B][H]; S0: fp32 [nb][H][D][D];
 *   n_acc: int32 [nb]; path: int32 [nb][B]; S_out: fp64 [nb][H][D][D]. */
int tvo_gdn_commit(const uint16_t *k, const uint16_t *v, const float *alpha, const float *beta, const float *S0,
                   const int32_t *n_acc, const int32_t *path, int nb, int B, int H, int D, double *S_out)
{
    if (!k || !v || !alpha || !beta || !S0 || !n_acc || !path || !S_out || nb < 0 || B < 1 || H < 1 || D < 1)
        return TVO_ERR_ARG;
    double *kk = malloc(sizeof(double) * (size_t)D * 3);
    if (!kk) return TVO_ERR_ARG;
    double *vv = kk + D, *ks = kk + 2 * D;
    int rc = TVO_OK;
    for (int b = 0; b < nb && rc == TVO_OK; b++) {
        const int n = n_acc[b];
        const int32_t *pr = path + (size_t)b * B;
        if (n < 0 || n >= B || pr[0] != 0) { rc = TVO_ERR_ARG; break; }
        for (int t = 1; t <= n; t++)
            if (pr[t] <= pr[t - 1] || pr[t] >= B) rc = TVO_ERR_ARG;
        if (rc != TVO_OK) break;
        for (int h = 0; h < H; h++) {
            double *S = S_out + ((size_t)b * H + h) * D * D;
            const float *s0 = S0 + ((size_t)b * H + h) * D * D;
            for (int x = 0; x < D * D; x++) S[x] = s0[x];
            for (int t = 0; t <= n; t++) {
                const size_t row = ((size_t)b * B + pr[t]) * H + h;
                const double a = alpha[row], be = beta[row];
                for (int d = 0; d < D; d++) { kk[d] = bf16_value(k[row * D + d]); vv[d] = bf16_value(v[row * D + d]); }
                for (int c = 0; c < D; c++) {            /* ks = k^T S */
                    double acc = 0.0;
                    for (int r = 0; r < D; r++) acc += kk[r] * S[(size_t)r * D + c];
                    ks[c] = acc;
                }
                for (int r = 0; r < D; r++)
                    for (int c = 0; c < D; c++)
                        S[(size_t)r * D + c] = a * (S[(size_t)r * D + c] - be * kk[r] * ks[c]) + be * kk[r] * vv[c];
            }
        }
    }
    free(kk);
    return rc;
}
