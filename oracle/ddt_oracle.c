/*
 * ddt_oracle.c -- plain CPU oracle for the DDTree verify step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this file's library.  It shares
 * no code, header, table or helper with the CUDA path; the two meet only at
 * the plain arrays produced by the seeded input generator.
 *
 * Everything here is written for a reader checking it against the pages by
 * eye: no blocking, no fusion, fp64 for all attention arithmetic.  Where the
 * pages fix no precision for the tree scores, they are summed in fp32 in
 * root-to-leaf order (the drafter hands over fp32 log-probs), because those
 * sums decide an integer outcome (which node is popped) and both sides must
 * take that decision in the same precision.
 *
 * Sources (page title, then section):
 *   [TREE]  "The DDTree CUDA Graph Fix: Unlocking Speculative Decoding at
 *           109 tok/s on PCIe Blackwell", section "The DDTree Architecture:
 *           Confirming Multiple-Path Evaluation" -- best-first heap expansion
 *           (pop the best cumulative log-prob node, push its best child and
 *           next sibling, stop at budget nodes; the tree has budget+1 nodes),
 *           visibility = ancestors plus the shared prefix, greedy accept walk
 *           returning the longest accepted chain plus one bonus token.
 *   [KV]    "The Architecture of a Speculative Decoding Engine", sections
 *           "The Final Resolution: A Concrete Trace" (root at position L,
 *           drafts attend to the cache plus their ancestor chain, the cache
 *           grows by accept_len) and "The Forward Pass Pseudocode" (absorbed
 *           MLA: scores over the 512 latent + 64 rope dims, output in the
 *           512-dim latent space).
 *   [MASK]  "The 30-Column Mask", sections "The Message: Tensor Shapes as
 *           Evidence", "The Fix: Building Combined Indices" and "Mask Stride
 *           Formula" -- kv columns are prefix slots followed by the tree
 *           nodes' slots, one mask row spans prefix + q_len columns.
 *   [ACC]   "The Oracle Drafter", section "The Engine Interface Design" --
 *           accept produces the accepted path, its length, the commit tokens
 *           and the bonus token.
 *   [SAMPLE] "The DDTree CUDA Graph Fix ...", section "Temperature Support:
 *           Already Working for Linear, Planned for DDTree" -- sampling accept
 *           reuses a tree rejection-sampling kernel that takes the tree as
 *           (retrieve_index, retrieve_next_token, retrieve_next_sibling) and
 *           filters the target with temperature, top-k and top-p.  The pages
 *           give no algorithm text; the reading taken is R15 below.
 *   [COMMIT] "The Architecture of a Speculative Decoding Engine", the
 *           append-then-compact scheme and "The Final Resolution: A Concrete
 *           Trace" -- every tree node's latent is appended after the
 *           committed prefix; after acceptance only the accepted nodes'
 *           latents are gathered into contiguous positions and the cache
 *           grows by accept_len.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes):
 *   R1  heap order: score descending, then depth ascending, then the path of
 *       sibling ranks compared lexicographically ascending.
 *   R2  scores: fp32, child = parent_score + logp[depth-1][rank].
 *   R3  kv column P_b + j is tree node j.
 *   R4  keys are the full 576-wide row, values its first 512 entries.
 *   R5  bit-packed mask: W_b = ceil((P_b+T_b)/32) uint32 words per row, bit
 *       (c mod 32) of word c/32, rows contiguous, request b starting at word
 *       mask_indptr[b] = sum over earlier requests of T*W.
 *   R6  among children of the current node, the first (lowest index) whose
 *       token equals the target's argmax is followed.
 *   R7  a row with no visible column gives out = 0 and lse = -inf.
 *   R8  accept_len counts the root; commit tokens = accepted drafts + bonus.
 *   R15 sampling accept (target-only, deterministic drafts): at node n the
 *       target distribution p is softmax(logits[n] / T) over the tokens whose
 *       logit is at least the top_k-th largest (all of them when top_k <= 0
 *       or >= vocab; ties kept).  Top-p then keeps the tokens whose logit is
 *       at least tau, the largest logit x with S(x) >= top_p, where S(x) is
 *       the mass of p over the tokens whose logit is at least x (the nucleus
 *       taken in logit order; tokens equal to tau are all kept), and p is
 *       renormalised over them; top_p outside (0, 1) keeps every token.
 *       The children of n are tried in index order
 *       against the residual r (p minus the tokens already rejected): child c
 *       with token t is taken when coin[n][i] < r(t) / mass(r), else t leaves
 *       the residual.  With no child taken, the bonus is the first token id v
 *       whose cumulative residual mass exceeds coin[n][last] * mass(r).  This
 *       emits every token with probability p, and T <= 0 (p = one-hot at the
 *       argmax, lowest id on ties) is the greedy walk exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_EXHAUSTED 2

#define OR_DL 512     /* latent width (values and first part of keys) */
#define OR_DR 64      /* rope width (second part of keys) */
#define OR_D 576      /* full key / query width */
#define OR_MAX_DEPTH 7

/* ------------------------------------------------------------------ */
/* Tree: best-first heap expansion over per-depth top-k     [TREE][R1][R2] */
/* ------------------------------------------------------------------ */

typedef struct {
    float score;              /* cumulative log-prob of this candidate (fp32) */
    float parent_score;       /* score of its parent (needed for the sibling) */
    int depth;                /* 1..max_depth */
    int rank;                 /* rank of this node among its parent's top-k */
    int ranks[OR_MAX_DEPTH];  /* path of ranks from the root, ranks[depth-1] == rank */
    int parent_out;           /* output index of the parent node */
} cand_t;

/* 1 if a should be popped before b (R1). */
static int cand_before(const cand_t *a, const cand_t *b) {
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    for (int d = 0; d < a->depth; ++d)
        if (a->ranks[d] != b->ranks[d]) return a->ranks[d] < b->ranks[d];
    return 0;
}

static void heap_push(cand_t *h, int *n, const cand_t *c) {
    int i = (*n)++;
    h[i] = *c;
    while (i > 0) {
        int p = (i - 1) / 2;
        if (!cand_before(&h[i], &h[p])) break;
        cand_t t = h[i]; h[i] = h[p]; h[p] = t;
        i = p;
    }
}

static cand_t heap_pop(cand_t *h, int *n) {
    cand_t top = h[0];
    h[0] = h[--(*n)];
    int i = 0;
    for (;;) {
        int l = 2 * i + 1, r = l + 1, best = i;
        if (l < *n && cand_before(&h[l], &h[best])) best = l;
        if (r < *n && cand_before(&h[r], &h[best])) best = r;
        if (best == i) break;
        cand_t t = h[i]; h[i] = h[best]; h[best] = t;
        i = best;
    }
    return top;
}

/*
 * topk_logp [B][max_depth][K] fp32, non-increasing along K (a drafter's top-k);
 * topk_ids  [B][max_depth][K]; root_id [B]; budget [B];
 * qo_indptr [B+1] with qo_indptr[b+1]-qo_indptr[b] == budget[b]+1.
 * Writes node_token / parent / depth, ragged by qo_indptr.  Node 0 of each
 * request is the root (token root_id, parent -1, depth 0); node n >= 1 is the
 * n-th pop.  Returns OR_ERR_EXHAUSTED if the implicit tree has fewer than
 * budget nodes.
 */
int oracle_build_tree(const float *topk_logp, const int32_t *topk_ids,
                      const int32_t *root_id, const int32_t *budget,
                      const int32_t *qo_indptr, int B, int max_depth, int K,
                      int32_t *node_token, int32_t *parent, int32_t *depth) {
    if (B < 0 || max_depth < 1 || max_depth > OR_MAX_DEPTH || K < 1) return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        const float *lp = topk_logp + (size_t)b * max_depth * K;
        const int32_t *ids = topk_ids + (size_t)b * max_depth * K;
        int base = qo_indptr[b];
        if (budget[b] < 0 || qo_indptr[b + 1] - base != budget[b] + 1) return OR_ERR_ARG;
        for (int d = 0; d < max_depth; ++d)
            for (int r = 1; r < K; ++r)
                if (!(lp[d * K + r] <= lp[d * K + r - 1])) return OR_ERR_ARG;

        node_token[base] = root_id[b];
        parent[base] = -1;
        depth[base] = 0;
        if (budget[b] == 0) continue;

        /* every pop adds at most one entry net, so budget+1 slots suffice */
        cand_t *heap = (cand_t *)malloc(sizeof(cand_t) * (size_t)(budget[b] + 2));
        int hn = 0;
        cand_t first;
        memset(&first, 0, sizeof first);
        first.parent_score = 0.0f;
        first.score = first.parent_score + lp[0];
        first.depth = 1;
        first.rank = 0;
        first.ranks[0] = 0;
        first.parent_out = 0;
        heap_push(heap, &hn, &first);

        int count = 0;
        while (count < budget[b] && hn > 0) {
            cand_t c = heap_pop(heap, &hn);
            int out = 1 + count;
            node_token[base + out] = ids[(c.depth - 1) * K + c.rank];
            parent[base + out] = c.parent_out;
            depth[base + out] = c.depth;
            ++count;
            if (c.depth < max_depth) {          /* best child of the popped node */
                cand_t ch = c;
                ch.parent_score = c.score;
                ch.score = c.score + lp[c.depth * K + 0];
                ch.depth = c.depth + 1;
                ch.rank = 0;
                ch.ranks[c.depth] = 0;
                ch.parent_out = out;
                heap_push(heap, &hn, &ch);
            }
            if (c.rank + 1 < K) {               /* next sibling of the popped node */
                cand_t sb = c;
                sb.rank = c.rank + 1;
                sb.ranks[c.depth - 1] = sb.rank;
                sb.score = c.parent_score + lp[(c.depth - 1) * K + sb.rank];
                heap_push(heap, &hn, &sb);
            }
        }
        free(heap);
        if (count < budget[b]) return OR_ERR_EXHAUSTED;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Visibility mask                                      [TREE][MASK][R3][R5] */
/* ------------------------------------------------------------------ */

/* mask_indptr[b] = word offset of request b (R5); mask_indptr[B] = total words. */
int oracle_mask_indptr(const int32_t *qo_indptr, const int32_t *prefix_len, int B,
                       int64_t *mask_indptr) {
    int64_t off = 0;
    for (int b = 0; b < B; ++b) {
        int64_t T = qo_indptr[b + 1] - qo_indptr[b];
        int64_t N = (int64_t)prefix_len[b] + T;
        if (T < 1 || prefix_len[b] < 0) return OR_ERR_ARG;
        mask_indptr[b] = off;
        off += T * ((N + 31) / 32);
    }
    mask_indptr[B] = off;
    return OR_OK;
}

/* Row i of request b: columns [0, P_b) are the shared prefix (all visible);
 * column P_b + j is visible iff node j is node i or one of its ancestors. */
int oracle_compile_visibility(const int32_t *parent, const int32_t *qo_indptr,
                              const int32_t *prefix_len, const int64_t *mask_indptr,
                              int B, uint32_t *mask) {
    for (int b = 0; b < B; ++b) {
        int T = qo_indptr[b + 1] - qo_indptr[b];
        int P = prefix_len[b];
        int64_t N = (int64_t)P + T;
        int64_t W = (N + 31) / 32;
        const int32_t *par = parent + qo_indptr[b];
        for (int i = 0; i < T; ++i) {
            uint32_t *row = mask + mask_indptr[b] + (int64_t)i * W;
            for (int64_t w = 0; w < W; ++w) row[w] = 0u;
            for (int64_t c = 0; c < P; ++c) row[c / 32] |= 1u << (c % 32);
            int guard = 0;
            for (int j = i; j >= 0; j = par[j]) {   /* self, then each ancestor */
                if (j >= T || ++guard > T) return OR_ERR_ARG;
                int64_t c = (int64_t)P + j;
                row[c / 32] |= 1u << (c % 32);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Tree-verify attention in absorbed MLA form, fp64          [KV][MASK][R4] */
/* ------------------------------------------------------------------ */

static double bf16_to_double(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * q [total_q][H][576] bf16 bits; kv_pool [pool_rows][576] bf16 bits;
 * kv_indices ragged by kv_indptr (prefix slots, then the T_b tree slots in node
 * order); mask as produced above.  For each requested row index
 * rows[r] = t*H + h it writes out[r][0:512] and lse[r] (natural log).
 */
int oracle_verify_attn(const uint16_t *q, const uint16_t *kv_pool, int64_t pool_rows,
                       const int32_t *kv_indices, const int32_t *kv_indptr,
                       const int32_t *qo_indptr, const uint32_t *mask,
                       const int64_t *mask_indptr, int B, int H, double scale,
                       const int64_t *rows, int64_t n_rows, double *out, double *lse,
                       int nthreads) {
    int64_t total_q = qo_indptr[B];
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= total_q * H) return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int T = qo_indptr[b + 1] - qo_indptr[b];
        int N = kv_indptr[b + 1] - kv_indptr[b];
        if (T < 1 || N < T) return OR_ERR_ARG;
        for (int j = 0; j < N; ++j) {
            int32_t s = kv_indices[kv_indptr[b] + j];
            if (s < 0 || s >= pool_rows) return OR_ERR_ARG;
        }
    }
    /* the thread count for this call only (0: all of OpenMP's default) */
#ifdef _OPENMP
    int team = nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    int team = 1;
    (void)nthreads;
#endif
    (void)team;

#pragma omp parallel for schedule(dynamic, 1) num_threads(team)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t t = rows[r] / H;
        int h = (int)(rows[r] % H);
        int b = 0;
        while (qo_indptr[b + 1] <= t) ++b;
        int i = (int)(t - qo_indptr[b]);
        int T = qo_indptr[b + 1] - qo_indptr[b];
        int N = kv_indptr[b + 1] - kv_indptr[b];
        int64_t W = (N + 31) / 32;
        const uint32_t *mrow = mask + mask_indptr[b] + (int64_t)i * W;
        const uint16_t *qrow = q + ((size_t)t * H + h) * OR_D;
        (void)T;

        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        double m = -INFINITY;
        for (int j = 0; j < N; ++j) {
            if (!((mrow[j / 32] >> (j % 32)) & 1u)) { s[j] = -INFINITY; continue; }
            const uint16_t *krow = kv_pool + (size_t)kv_indices[kv_indptr[b] + j] * OR_D;
            double dot = 0.0;
            for (int d = 0; d < OR_D; ++d) dot += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double *o = out + (size_t)r * OR_DL;
        for (int d = 0; d < OR_DL; ++d) o[d] = 0.0;
        if (m == -INFINITY) {           /* R7: nothing visible */
            lse[r] = -INFINITY;
            free(s);
            continue;
        }
        double denom = 0.0;
        for (int j = 0; j < N; ++j) {
            if (s[j] == -INFINITY) continue;
            double w = exp(s[j] - m);
            denom += w;
            const uint16_t *vrow = kv_pool + (size_t)kv_indices[kv_indptr[b] + j] * OR_D;
            for (int d = 0; d < OR_DL; ++d) o[d] += w * bf16_to_double(vrow[d]);
        }
        for (int d = 0; d < OR_DL; ++d) o[d] /= denom;
        lse[r] = m + log(denom);
        free(s);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Greedy accept walk                                  [TREE][ACC][KV][R6][R8] */
/* ------------------------------------------------------------------ */

/*
 * accepted_nodes and commit_tokens are [B][max_depth+1], padded with -1.
 * accept_len[b] = number of accepted nodes including the root; the commit
 * tokens are the accepted draft tokens followed by the bonus token (the
 * target's argmax at the last accepted node), accept_len tokens in all.
 */
int oracle_accept(const int32_t *node_token, const int32_t *parent,
                  const int32_t *qo_indptr, const int32_t *target_argmax, int B,
                  int max_depth, int32_t *accept_len, int32_t *accepted_nodes,
                  int32_t *commit_tokens, int32_t *bonus) {
    int width = max_depth + 1;
    for (int b = 0; b < B; ++b) {
        int base = qo_indptr[b];
        int T = qo_indptr[b + 1] - base;
        int32_t *acc = accepted_nodes + (size_t)b * width;
        int32_t *com = commit_tokens + (size_t)b * width;
        for (int k = 0; k < width; ++k) { acc[k] = -1; com[k] = -1; }
        int cur = 0, n = 0;
        acc[n++] = 0;
        for (;;) {
            int want = target_argmax[base + cur];
            int next = -1;
            for (int c = 1; c < T; ++c)
                if (parent[base + c] == cur && node_token[base + c] == want) { next = c; break; }
            if (next < 0) break;
            if (n >= width) return OR_ERR_ARG;   /* deeper than max_depth */
            acc[n++] = next;
            cur = next;
        }
        accept_len[b] = n;
        bonus[b] = target_argmax[base + cur];
        for (int k = 1; k < n; ++k) com[k - 1] = node_token[base + acc[k]];
        com[n - 1] = bonus[b];
    }
    return OR_OK;
}

/*
 * [COMMIT] Gather the accepted latents of request b into positions
 * P_b .. P_b + accept_len - 1 of its sequence (position c lives in pool row
 * kv_indices[kv_indptr[b] + c]).  All source rows are copied out first, then
 * written, so the result is "the accepted nodes' original latents in path
 * order" whatever the overlap between sources and destinations.  new_len[b]
 * = P_b + accept_len[b].  Returns OR_ERR_ARG (and changes nothing for that
 * request) if the accepted path is not 0 = a_0 < a_1 < ... < q_len or a row
 * is outside the pool.
 */
int oracle_commit_kv(uint16_t *kv_pool, int64_t pool_rows, const int32_t *kv_indices,
                     const int32_t *kv_indptr, const int32_t *qo_indptr,
                     const int32_t *accept_len, const int32_t *accepted_nodes, int B,
                     int max_depth, int32_t *new_len) {
    const int D = 576;
    int width = max_depth + 1;
    int status = OR_OK;
    uint16_t *tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)width * D);
    if (!tmp) return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int T = qo_indptr[b + 1] - qo_indptr[b];
        int N = kv_indptr[b + 1] - kv_indptr[b];
        int P = N - T;
        int n = accept_len[b];
        const int32_t *acc = accepted_nodes + (size_t)b * width;
        const int32_t *idx = kv_indices + kv_indptr[b];
        int ok = n >= 1 && n <= width && n <= T && acc[0] == 0;
        for (int k = 1; ok && k < n; ++k)
            if (acc[k] <= acc[k - 1] || acc[k] >= T) ok = 0;
        for (int k = 0; ok && k < n; ++k) {
            int64_t src = idx[P + acc[k]], dst = idx[P + k];
            if (src < 0 || src >= pool_rows || dst < 0 || dst >= pool_rows) ok = 0;
        }
        if (!ok) { status = OR_ERR_ARG; continue; }
        for (int k = 0; k < n; ++k)
            memcpy(tmp + (size_t)k * D, kv_pool + (size_t)idx[P + acc[k]] * D, sizeof(uint16_t) * D);
        for (int k = 0; k < n; ++k)
            memcpy(kv_pool + (size_t)idx[P + k] * D, tmp + (size_t)k * D, sizeof(uint16_t) * D);
        if (new_len) new_len[b] = P + n;
    }
    free(tmp);
    return status;
}

/*
 * [SAMPLE] The tree in the sampling kernel's format: for node n of request b,
 * retrieve_index[n] = qo_indptr[b] + n (its row), first_child[n] = the lowest
 * index child of n or -1 (retrieve_next_token), next_sibling[n] = the next
 * higher index child of n's parent or -1 (retrieve_next_sibling).  Indices
 * other than retrieve_index are local to the request.
 */
int oracle_tree_links(const int32_t *parent, const int32_t *qo_indptr, int B,
                      int32_t *first_child, int32_t *next_sibling, int32_t *retrieve_index) {
    for (int b = 0; b < B; ++b) {
        int base = qo_indptr[b];
        int T = qo_indptr[b + 1] - base;
        for (int n = 0; n < T; ++n) {
            first_child[base + n] = -1;
            next_sibling[base + n] = -1;
            retrieve_index[base + n] = base + n;
        }
        for (int c = 1; c < T; ++c) {
            int p = parent[base + c];
            if (p < 0 || p >= c) return OR_ERR_ARG;
            if (first_child[base + p] < 0) {
                first_child[base + p] = c;
            } else {
                int s = first_child[base + p];
                while (next_sibling[base + s] >= 0) s = next_sibling[base + s];
                next_sibling[base + s] = c;
            }
        }
    }
    return OR_OK;
}

static int cmp_desc(const void *a, const void *b) {
    float x = *(const float *)a, y = *(const float *)b;
    return (x < y) - (x > y);
}

/*
 * [SAMPLE] reading R15.  coins is [rows][coin_stride] uniform [0,1): coin i is
 * for the i-th child tried at that node, the last one for the bonus draw.
 * top_p is [B] or NULL (no top-p).  Outputs as in oracle_accept.
 */
int oracle_accept_sampled(const int32_t *node_token, const int32_t *parent,
                          const int32_t *qo_indptr, const float *logits, int vocab,
                          const float *temperature, const int32_t *top_k, const float *top_p,
                          const float *coins, int coin_stride, int B, int max_depth,
                          int32_t *accept_len, int32_t *accepted_nodes, int32_t *commit_tokens,
                          int32_t *bonus) {
    int width = max_depth + 1;
    double *p = (double *)malloc(sizeof(double) * (size_t)vocab);
    float *sorted = (float *)malloc(sizeof(float) * (size_t)vocab);
    if (!p || !sorted) { free(p); free(sorted); return OR_ERR_ARG; }
    int status = OR_OK;
    for (int b = 0; b < B && status == OR_OK; ++b) {
        int base = qo_indptr[b];
        int T = qo_indptr[b + 1] - base;
        int32_t *acc = accepted_nodes + (size_t)b * width;
        int32_t *com = commit_tokens + (size_t)b * width;
        for (int k = 0; k < width; ++k) { acc[k] = -1; com[k] = -1; }
        int cur = 0, n = 0;
        acc[n++] = 0;
        for (;;) {
            const float *l = logits + (size_t)(base + cur) * vocab;
            const float *u = coins + (size_t)(base + cur) * coin_stride;
            /* the target distribution p at this node */
            int amax = 0;
            for (int v = 1; v < vocab; ++v) if (l[v] > l[amax]) amax = v;
            if (temperature[b] <= 0.0f) {
                for (int v = 0; v < vocab; ++v) p[v] = (v == amax) ? 1.0 : 0.0;
            } else {
                float thr = -INFINITY;
                int k = top_k[b];
                if (k > 0 && k < vocab) {
                    memcpy(sorted, l, sizeof(float) * (size_t)vocab);
                    qsort(sorted, (size_t)vocab, sizeof(float), cmp_desc);
                    thr = sorted[k - 1];
                }
                double z = 0.0;
                for (int v = 0; v < vocab; ++v) {
                    p[v] = (l[v] >= thr) ? exp(((double)l[v] - (double)l[amax]) / (double)temperature[b]) : 0.0;
                    z += p[v];
                }
                for (int v = 0; v < vocab; ++v) p[v] /= z;
                double tp = top_p ? (double)top_p[b] : 1.0;
                if (tp > 0.0 && tp < 1.0) {
                    /* the kept logits in descending order; walk groups of equal
                       logits, adding their mass, until the mass reaches top_p */
                    int m = 0;
                    for (int v = 0; v < vocab; ++v) if (l[v] >= thr) sorted[m++] = l[v];
                    qsort(sorted, (size_t)m, sizeof(float), cmp_desc);
                    double S = 0.0;
                    float tau = sorted[m - 1];
                    for (int i = 0; i < m;) {
                        float x = sorted[i];
                        double px = exp(((double)x - (double)l[amax]) / (double)temperature[b]) / z;
                        int j = i;
                        while (j < m && sorted[j] == x) { S += px; ++j; }
                        if (S >= tp) { tau = x; break; }
                        i = j;
                    }
                    double z2 = 0.0;
                    for (int v = 0; v < vocab; ++v) {
                        if (l[v] < tau) p[v] = 0.0;
                        z2 += p[v];
                    }
                    for (int v = 0; v < vocab; ++v) p[v] /= z2;
                }
            }
            /* the children, in index order, against the residual; a node needs
               one coin per child plus one for the bonus */
            int nkids = 0;
            for (int c = 1; c < T; ++c) nkids += parent[base + c] == cur;
            if (nkids > coin_stride - 1) { status = OR_ERR_ARG; break; }
            double mass = 1.0;
            int next = -1, tried = 0;
            for (int c = 1; c < T; ++c) {
                if (parent[base + c] != cur) continue;
                int t = node_token[base + c];
                double pt = (t >= 0 && t < vocab) ? p[t] : 0.0;
                if ((double)u[tried] < pt / mass) { next = c; break; }
                if (t >= 0 && t < vocab) { mass -= pt; p[t] = 0.0; }
                ++tried;
            }
            if (status != OR_OK) break;
            if (next >= 0) {
                if (n >= width) { status = OR_ERR_ARG; break; }   /* deeper than max_depth */
                acc[n++] = next;
                cur = next;
                continue;
            }
            /* bonus: inverse CDF of the residual in token-id order */
            double target = (double)u[coin_stride - 1] * mass, cum = 0.0;
            int bon = -1, last = -1;
            for (int v = 0; v < vocab; ++v) {
                if (p[v] <= 0.0) continue;
                last = v;
                cum += p[v];
                if (cum > target) { bon = v; break; }
            }
            if (bon < 0) bon = (last >= 0) ? last : amax;
            accept_len[b] = n;
            bonus[b] = bon;
            for (int k = 1; k < n; ++k) com[k - 1] = node_token[base + acc[k]];
            com[n - 1] = bon;
            break;
        }
    }
    free(p);
    free(sorted);
    return status;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
