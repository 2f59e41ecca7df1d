/*
 * jf_oracle.c -- plain, slow fp64 CPU oracle for tree-causal paged attention and
 * greedy tree verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header or table with the
 * CUDA path (tree_speculative_decoding_jf_gb300/csrc) and never calls it.
 *
 * Every function follows a definition from the JetFlow explainer pages ("JetFlow:
 * Breaking the Scaling Ceiling of Speculative Decoding with Parallel Tree Drafting",
 * gist.science explainer, technical summary §2 "Method" and §4 "Results"; qxai.app
 * commentary, section "まず、何が問題なのか").  Where the pages leave a step open the
 * plainest reading is taken; each reading is named where it is used.
 *
 * Floating point: every score, weight and sum is a double.  bf16 inputs are widened
 * exactly (bits << 16 is the fp32 value, which a double holds exactly).
 *
 * Parity status: mask, attention, argmax and tree walk are all pinned by the CPU test
 * suite (brute force, closed forms, library special cases); the greedy acceptance rule
 * itself is a reading of "the target keeps the drafted prefix it agrees with" and is
 * not fixed more precisely by the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define JFO_OK 0
#define JFO_BAD_TREE 2
#define JFO_BAD_ARG 1

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* A tree is valid when parent[0] == -1 and 0 <= parent[i] < i for i >= 1
 * (nodes are numbered in topological order, root first). */
static int tree_is_valid(const int32_t *parent, int N) {
    if (N < 1 || parent[0] != -1) return 0;
    for (int i = 1; i < N; ++i)
        if (parent[i] < 0 || parent[i] >= i) return 0;
    return 1;
}

/* anc(i) = {i} u anc(parent[i]), anc(root) = {root}.  Tree-causal mask: a node sees
 * its own ancestors in the draft tree (and itself), never descendants or unrelated
 * sibling branches (JetFlow explainer §2, "Tree-Causal Attention Mask").  The member
 * flags are written into is_anc[0..N). */
static void ancestor_set(const int32_t *parent, int N, int i, unsigned char *is_anc) {
    memset(is_anc, 0, (size_t)N);
    for (int a = i; a >= 0; a = parent[a]) is_anc[a] = 1;
}

/* Packed ancestor-or-self bitmask per node: bit (j & 63) of word (j >> 6) of row i is
 * set iff j in anc(i); padding bits are 0.  depth[i] = |anc(i)| - 1 and
 * pos[i] = prefix_len[b] + depth[i] (the root sits right after the prefix).
 * Returns JFO_BAD_TREE if any tree is not in topological order. */
int jfo_tree_mask(const int32_t *parent, const int32_t *prefix_len, int B, int N,
                  uint64_t *mask, int32_t *depth, int32_t *pos) {
    const int W = (N + 63) / 64;
    unsigned char *is_anc = (unsigned char *)malloc((size_t)N);
    if (!is_anc) return JFO_BAD_ARG;
    int rc = JFO_OK;
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (size_t)b * N;
        if (!tree_is_valid(par, N)) { rc = JFO_BAD_TREE; continue; }
        for (int i = 0; i < N; ++i) {
            ancestor_set(par, N, i, is_anc);
            uint64_t *row = mask + ((size_t)b * N + i) * W;
            int count = 0;
            for (int w = 0; w < W; ++w) row[w] = 0;
            for (int j = 0; j < N; ++j)
                if (is_anc[j]) {
                    row[j >> 6] |= (uint64_t)1 << (j & 63);
                    ++count;
                }
            depth[(size_t)b * N + i] = count - 1;
            pos[(size_t)b * N + i] = prefix_len[b] + count - 1;
        }
    }
    free(is_anc);
    return rc;
}

/* Key t of sequence b, kv-head g: logical position t lives in page
 * block_table[b][t / page], slot t % page, of a pool laid out
 * [num_pages][page][Hkv][D] (paged KV cache; explainer §3 names the paged kernel). */
static const uint16_t *paged_row(const uint16_t *cache, const int32_t *bt_row, int page,
                                 int Hkv, int D, int g, long t) {
    long pg = bt_row[t / page];
    long slot = t % page;
    return cache + ((pg * page + slot) * Hkv + g) * (long)D;
}

/* One query row (b, h, i) of tree-causal attention.
 *   visible keys S = {0..P_b-1} u {P_b + j : j in anc(i)}   (prefix + own root path)
 *   s_t = scale * q . k_t ;  m = max s ;  w_t = exp(s_t - m)
 *   out = sum_t w_t v_t / sum_t w_t ;  lse = m + log(sum_t w_t)
 * Keys outside S are never touched, so their weight is exactly zero (the branch
 * factorisation q(pi(v)|x) = prod_{u in pi(v)} q(y_u | x, h_x, pi_{<u}) of explainer
 * §2 conditions each node on the prefix and its own path only).
 * Reading: tree node j's K/V sit at logical position P_b + j of the same paged cache. */
static void attention_row(const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                          const int32_t *bt, const int32_t *prefix_len,
                          const int32_t *parent, int N, int Hq, int Hkv, int D, int page,
                          int max_pages, double scale, int b, int h, int i,
                          double *out, double *lse, double *probs_row,
                          unsigned char *is_anc, double *qd, double *s) {
    const int G = Hq / Hkv;
    const int g = h / G;
    const long P = prefix_len[b];
    const int32_t *par = parent + (size_t)b * N;
    const int32_t *bt_row = bt + (size_t)b * max_pages;
    ancestor_set(par, N, i, is_anc);
    const uint16_t *qrow = q + (((size_t)b * N + i) * Hq + h) * (size_t)D;
    for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(qrow[d]);

    const long L = P + N;
    double m = -INFINITY;
    for (long t = 0; t < L; ++t) {
        int visible = (t < P) || is_anc[t - P];
        if (!visible) { s[t] = -INFINITY; continue; }
        const uint16_t *k = paged_row(kc, bt_row, page, Hkv, D, g, t);
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qd[d] * bf16_to_double(k[d]);
        s[t] = scale * acc;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (long t = 0; t < L; ++t) {
        int visible = (t < P) || is_anc[t - P];
        if (!visible) { if (probs_row) probs_row[t] = 0.0; continue; }
        double w = exp(s[t] - m);
        s[t] = w;
        l += w;
        const uint16_t *v = paged_row(vc, bt_row, page, Hkv, D, g, t);
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_double(v[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    if (probs_row)
        for (long t = 0; t < L; ++t) {
            int visible = (t < P) || is_anc[t - P];
            if (visible) probs_row[t] = s[t] / l;
        }
    *lse = m + log(l);
}

/* Tree-causal paged attention for a list of query rows (b, h, i).
 * out: double [nrows][D]; lse: double [nrows].  The rows may be every (b, h, i) of
 * the problem or a sample of them.  Returns JFO_BAD_TREE on an invalid tree. */
int jfo_tree_attention_rows(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_table,
                            const int32_t *prefix_len, const int32_t *parent, int B, int N,
                            int Hq, int Hkv, int D, int page, int max_pages, double scale,
                            long nrows, const int32_t *rows_b, const int32_t *rows_h,
                            const int32_t *rows_i, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || page <= 0) return JFO_BAD_ARG;
    for (int b = 0; b < B; ++b)
        if (!tree_is_valid(parent + (size_t)b * N, N)) return JFO_BAD_TREE;
    long Lmax = 0;
    for (int b = 0; b < B; ++b)
        if (prefix_len[b] + N > Lmax) Lmax = prefix_len[b] + N;
    int rc = JFO_OK;
#pragma omp parallel
    {
        unsigned char *is_anc = (unsigned char *)malloc((size_t)N);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
        if (!is_anc || !qd || !s) {
#pragma omp atomic write
            rc = JFO_BAD_ARG;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < nrows; ++r)
                attention_row(q, k_cache, v_cache, block_table, prefix_len, parent, N, Hq,
                              Hkv, D, page, max_pages, scale, rows_b[r], rows_h[r],
                              rows_i[r], out + r * (long)D, lse + r, NULL, is_anc, qd, s);
        }
        free(is_anc);
        free(qd);
        free(s);
    }
    return rc;
}

/* Full probability matrix of one (b, h): probs [N][P_b + N], zero where masked.
 * Small inputs only (inspection of the mask's effect on the weights). */
int jfo_attention_probs(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_table, const int32_t *prefix_len,
                        const int32_t *parent, int B, int N, int Hq, int Hkv, int D,
                        int page, int max_pages, double scale, int b, int h,
                        double *probs) {
    if (b < 0 || b >= B) return JFO_BAD_ARG;
    if (!tree_is_valid(parent + (size_t)b * N, N)) return JFO_BAD_TREE;
    const long L = prefix_len[b] + N;
    unsigned char *is_anc = (unsigned char *)malloc((size_t)N);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    double *out = (double *)malloc(sizeof(double) * (size_t)D);
    double lse;
    for (int i = 0; i < N; ++i)
        attention_row(q, k_cache, v_cache, block_table, prefix_len, parent, N, Hq, Hkv, D,
                      page, max_pages, scale, b, h, i, out, &lse, probs + (long)i * L, is_anc,
                      qd, s);
    free(is_anc); free(qd); free(s); free(out);
    return JFO_OK;
}

/* argmax over a row compared as real numbers; the lowest index wins a tie, and
 * -0 equals +0 (double comparison).  The target's greedy choice per tree node
 * (reading of "the target model checks the drafts", qxai.app commentary). */
int jfo_argmax_f32(const float *logits, long rows, long V, int32_t *out) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const float *x = logits + r * V;
        long best = 0;
        double bv = (double)x[0];
        for (long v = 1; v < V; ++v)
            if ((double)x[v] > bv) { bv = (double)x[v]; best = v; }
        out[r] = (int32_t)best;
    }
    return JFO_OK;
}

int jfo_argmax_bf16(const uint16_t *logits, long rows, long V, int32_t *out) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const uint16_t *x = logits + r * V;
        long best = 0;
        double bv = bf16_to_double(x[0]);
        for (long v = 1; v < V; ++v) {
            double xv = bf16_to_double(x[v]);
            if (xv > bv) { bv = xv; best = v; }
        }
        out[r] = (int32_t)best;
    }
    return JFO_OK;
}

/* len(i) = 0 if node i has no accepted child, else 1 + max len(c) over accepted
 * children c.  A child c of p is accepted iff draft[c] == argmax[p] (greedy reading of
 * "keep the drafted prefix the target agrees with"). */
static int accepted_len(const int32_t *argmax, const int32_t *draft, const int32_t *parent,
                        int N, int i) {
    int best = 0;
    for (int c = i + 1; c < N; ++c)
        if (parent[c] == i && draft[c] == argmax[i]) {
            int l = 1 + accepted_len(argmax, draft, parent, N, c);
            if (l > best) best = l;
        }
    return best;
}

/* Greedy tree verification: accept_len = len(root) (draft nodes accepted, root not
 * counted); path = root, then repeatedly the accepted child with the greatest len
 * (ties: smallest node id), padded with -1; bonus = argmax at the path's last node.
 * Returns JFO_BAD_TREE on an invalid tree. */
int jfo_tree_walk(const int32_t *argmax, const int32_t *draft, const int32_t *parent, int B,
                  int N, int32_t *accept_len, int32_t *path, int32_t *bonus) {
    int rc = JFO_OK;
    for (int b = 0; b < B; ++b) {
        const int32_t *am = argmax + (size_t)b * N;
        const int32_t *dr = draft + (size_t)b * N;
        const int32_t *par = parent + (size_t)b * N;
        int32_t *pa = path + (size_t)b * N;
        if (!tree_is_valid(par, N)) { rc = JFO_BAD_TREE; continue; }
        for (int k = 0; k < N; ++k) pa[k] = -1;
        int cur = 0, n = 0;
        pa[n++] = 0;
        for (;;) {
            int best_c = -1, best_l = -1;
            for (int c = cur + 1; c < N; ++c)
                if (par[c] == cur && dr[c] == am[cur]) {
                    int l = accepted_len(am, dr, par, N, c);
                    if (l > best_l) { best_l = l; best_c = c; }
                }
            if (best_c < 0) break;
            cur = best_c;
            pa[n++] = cur;
        }
        accept_len[b] = n - 1;
        bonus[b] = am[cur];
    }
    return rc;
}

/* Accepted-path KV compaction (row "accepted-path KV compaction" after verification;
 * JetFlow explainer, technical summary §2 "Method": draft nodes keep their K/V after the
 * prefix, the accepted branch is the context the target continues from; the cache update
 * itself is not spelled out on the pages, so the plainest reading is taken).
 * For sequence b with a = accept_len[b] and P = prefix_len[b], for k = 1..a in order, the
 * K and V rows of every kv-head at logical position P + path[k] are copied to P + k;
 * new_prefix_len[b] = P + a + 1.  A sequence with a malformed prefix length, accepted
 * length, path (path[0] == 0, strictly increasing, inside [0, N)) or block-table entry is
 * left unchanged with new_prefix_len[b] = P; the function then returns JFO_BAD_ARG. */
int jfo_compact_accepted_kv(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_table,
                            const int32_t *prefix_len, const int32_t *path,
                            const int32_t *accept_len, int B, int N, int Hkv, int D, int page,
                            int max_pages, int num_pages, int32_t *new_prefix_len) {
    int rc = JFO_OK;
    for (int b = 0; b < B; ++b) {
        const int32_t *bt = block_table + (long)b * max_pages;
        const int32_t *pth = path + (long)b * N;
        const int P = prefix_len[b], a = accept_len[b];
        int ok = P >= 0 && (long)P + N <= (long)max_pages * page && a >= 0 && a <= N - 1;
        for (int k = 0; ok && k <= a; ++k) {
            if (k == 0 ? pth[0] != 0 : (pth[k] <= pth[k - 1] || pth[k] >= N)) ok = 0;
            else {
                const int ps = bt[(P + pth[k]) / page], pd = bt[(P + k) / page];
                if (ps < 0 || ps >= num_pages || pd < 0 || pd >= num_pages) ok = 0;
            }
        }
        new_prefix_len[b] = ok ? P + a + 1 : P;
        if (!ok) { rc = JFO_BAD_ARG; continue; }
        for (int k = 1; k <= a; ++k) {
            const int ts = P + pth[k], td = P + k;
            for (int g = 0; g < Hkv; ++g) {
                const long src = (((long)bt[ts / page] * page + ts % page) * Hkv + g) * D;
                const long dst = (((long)bt[td / page] * page + td % page) * Hkv + g) * D;
                for (int d = 0; d < D; ++d) {
                    k_cache[dst + d] = k_cache[src + d];
                    v_cache[dst + d] = v_cache[src + d];
                }
            }
        }
    }
    return rc;
}
