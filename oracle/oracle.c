/*
 * oracle.c - plain, slow, fp64 CPU oracle for tree-causal attention and
 * greedy tree verification.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg load this library. The product path
 * (the CUDA library and its Python binding) never calls it, and the two
 * share no code, headers, tables or constants.
 *
 * Sources (the method is JetFlow, arXiv 2606.18394; JetSpec on some pages):
 *  [blog]  "JetFlow: Scaling Speculative Decoding with Parallel Tree
 *          Drafting" (james.trappett.org), section "What JetFlow Does
 *          Differently". A tree node attends to the original prefix and to
 *          its own ancestors, never to siblings or descendants. A path's
 *          probability is a product of conditionals, each on the concrete
 *          ancestor tokens of that branch.
 *  [paper] Chinese translation of the paper (bittide.aicompass.dev),
 *          section 2.1 "Background". The target model verifies the N
 *          drafted tokens in parallel and accepts the longest prefix that
 *          agrees with its own predictions.
 *
 * Readings where the pages say nothing:
 *  - scale = 1/sqrt(head_dim) unless the caller passes another;
 *  - query head h uses KV head floor(h / (Hq/Hkv));
 *  - node 0 is the root (the last committed token); its own token is never
 *    checked; the logits of node u predict the children of u;
 *  - accept length counts path nodes including the root;
 *  - among accepted nodes of equal depth the lowest index wins;
 *  - argmax: ties go to the lowest index, +0 and -0 are equal, and NaN
 *    ranks above every number (the first NaN wins).
 *
 * Pins (tests/test_oracle_pins.py): torch fp64 scaled_dot_product_attention
 * with an independently built boolean mask; the chain tree equals textbook
 * causal attention; with q = 0 the output is the plain mean of the visible
 * values (closed form); relabelling or deleting non-ancestor nodes leaves a
 * node's output bit-identical; torch.argmax; brute-force path enumeration
 * on every tree with up to 6 nodes; hand-worked walk cases in
 * tests/golden/walk_cases.txt; hand-worked KV-commit cases in
 * tests/golden/commit_cases.txt. Stochastic verification
 * (tests/test_oracle_sample_pins.py): Philox4x64-10 word for word against
 * numpy's Philox generator; the emitted tokens' distribution equals the
 * target's (chi-square) when children are drawn from the draft, at the
 * root and one level down; draft = target accepts every first child; a
 * near-zero temperature with a flat draft gives the greedy walk. Path
 * scoring (tests/test_oracle_score_pins.py): torch.log_softmax gathered at
 * the tokens; an ancestor-indicator matrix built by transitive closure;
 * the frequency of drawing a path level by level; -depth ln V for uniform
 * logits; a stable descending torch.sort for the top-k; a brute-force sort
 * of every candidate for the budgeted expansion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact bf16 -> double: a bf16 is the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* A sequence's tree is well formed iff 1 <= n <= max_nodes, parents[0] = -1
 * and 0 <= parents[i] < i for 0 < i < n (topological order). */
int oracle_tree_is_valid(const int32_t *parents_b, int32_t n, int32_t max_nodes)
{
    if (n < 1 || n > max_nodes) return 0;
    if (parents_b[0] != -1) return 0;
    for (int32_t i = 1; i < n; ++i)
        if (parents_b[i] < 0 || parents_b[i] >= i) return 0;
    return 1;
}

/* Root-to-i ancestor chain (i included) of a well-formed tree; returns its
 * length. [blog] "each node can attend to the original prefix and its
 * ancestors in the tree". */
static int32_t ancestor_chain(const int32_t *parents_b, int32_t i, int32_t *chain)
{
    int32_t len = 0;
    for (int32_t j = i; j >= 0; j = parents_b[j]) chain[len++] = j;
    for (int32_t a = 0, z = len - 1; a < z; ++a, --z) {
        int32_t t = chain[a];
        chain[a] = chain[z];
        chain[z] = t;
    }
    return len;
}

/*
 * Tree attention, literally: for node i of sequence b the key/value sequence
 * is prefix[0 .. P_b) followed by the tree rows of i's ancestors, root first,
 * ending with i itself. Node i is the last query of ordinary causal attention
 * over that sequence ([blog]: the draft distribution along a branch is a
 * product of conditionals on that branch's concrete ancestors).
 *
 * q, out [B, Nmax, Hq, d]; k_cache, v_cache [B, Hkv, Pcap, d];
 * tree_k, tree_v [B, Nmax, Hkv, d]. All bf16 inputs are raw uint16 bits.
 * scale <= 0 selects 1/sqrt(d).
 * sel: n_sel (b, i) pairs to compute, or NULL for every (b, i) with
 *      i < n_nodes[b]. Rows not computed are left untouched.
 * A sequence whose tree or prefix length is malformed gets NaN in every
 * selected row.
 */
void oracle_tree_attention_f64(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                               const int32_t *prefix_lens, const uint16_t *tree_k,
                               const uint16_t *tree_v, const int32_t *parents,
                               const int32_t *n_nodes, int32_t B, int32_t Nmax, int32_t Hq,
                               int32_t Hkv, int32_t d, int32_t Pcap, double scale,
                               const int32_t *sel, int64_t n_sel, double *out)
{
    const int32_t G = Hq / Hkv;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)d);
    int64_t n_rows = sel ? n_sel : (int64_t)B * Nmax;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * ((size_t)Pcap + (size_t)Nmax));
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        int32_t *chain = (int32_t *)malloc(sizeof(int32_t) * (size_t)Nmax);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            int32_t b = sel ? sel[2 * r] : (int32_t)(r / Nmax);
            int32_t i = sel ? sel[2 * r + 1] : (int32_t)(r % Nmax);
            const int32_t *par = parents + (int64_t)b * Nmax;
            int32_t n = n_nodes[b];
            int32_t P = prefix_lens[b];
            int ok = oracle_tree_is_valid(par, n, Nmax) && P >= 0 && P <= Pcap;
            if (ok && i >= n) continue; /* padded node: not an output row */
            for (int32_t h = 0; h < Hq; ++h) {
                double *o = out + (((int64_t)b * Nmax + i) * Hq + h) * d;
                if (!ok) {
                    for (int32_t c = 0; c < d; ++c) o[c] = NAN;
                    continue;
                }
                int32_t kh = h / G;
                int32_t len = ancestor_chain(par, i, chain);
                const uint16_t *qv = q + (((int64_t)b * Nmax + i) * Hq + h) * d;
                const uint16_t *kc = k_cache + ((int64_t)b * Hkv + kh) * Pcap * d;
                const uint16_t *vc = v_cache + ((int64_t)b * Hkv + kh) * Pcap * d;
                int32_t L = P + len;
                /* scores s_j = scale * <q, k_j> over the causal sequence */
                for (int32_t j = 0; j < L; ++j) {
                    const uint16_t *kv = j < P ? kc + (int64_t)j * d
                                               : tree_k + (((int64_t)b * Nmax + chain[j - P]) * Hkv + kh) * d;
                    double dot = 0.0;
                    for (int32_t c = 0; c < d; ++c) dot += bf16_to_double(qv[c]) * bf16_to_double(kv[c]);
                    s[j] = scale * dot;
                }
                /* softmax over the sequence, then the weighted sum of values */
                double m = -INFINITY;
                for (int32_t j = 0; j < L; ++j) if (s[j] > m) m = s[j];
                double z = 0.0;
                for (int32_t c = 0; c < d; ++c) acc[c] = 0.0;
                for (int32_t j = 0; j < L; ++j) {
                    double w = exp(s[j] - m);
                    z += w;
                    const uint16_t *vv = j < P ? vc + (int64_t)j * d
                                               : tree_v + (((int64_t)b * Nmax + chain[j - P]) * Hkv + kh) * d;
                    for (int32_t c = 0; c < d; ++c) acc[c] += w * bf16_to_double(vv[c]);
                }
                for (int32_t c = 0; c < d; ++c) o[c] = acc[c] / z;
            }
        }
        free(s);
        free(acc);
        free(chain);
    }
}

/* First index of the maximum of one bf16 row: strict '>' keeps the first
 * of equal values (+0 == -0); a NaN ranks above every number, so the first
 * NaN is returned as soon as it is met. */
int32_t oracle_argmax_row(const uint16_t *row, int64_t V)
{
    double best = bf16_to_double(row[0]);
    int64_t arg = 0;
    if (isnan(best)) return 0;
    for (int64_t v = 1; v < V; ++v) {
        double x = bf16_to_double(row[v]);
        if (isnan(x)) return (int32_t)v;
        if (x > best) {
            best = x;
            arg = v;
        }
    }
    return (int32_t)arg;
}

/* argmax of n_rows rows of length V (row r at logits + r * V). */
void oracle_argmax_rows(const uint16_t *logits, int64_t n_rows, int64_t V, int32_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) out[r] = oracle_argmax_row(logits + r * V, V);
}

/* Naive recursion from the root: a child c of an accepted node u is accepted
 * iff tokens[c] equals the target's greedy prediction at u ([paper] 2.1). */
static void accept_from(int32_t u, int32_t depth, const int32_t *par, const int32_t *tok,
                        const int32_t *am, int32_t n, int32_t *best, int32_t *best_depth)
{
    if (depth > *best_depth || (depth == *best_depth && u < *best)) {
        *best = u;
        *best_depth = depth;
    }
    for (int32_t c = 0; c < n; ++c)
        if (par[c] == u && c != u && tok[c] == am[u])
            accept_from(c, depth + 1, par, tok, am, n, best, best_depth);
}

/*
 * Greedy tree verification for B sequences.
 * am[b, i] = argmax of logits row (b, i) for i < n_nodes[b]. The accepted
 * node is the deepest node whose every edge on the root path agrees
 * (lowest index on ties). The path runs root first, and accept_len counts
 * its nodes, root included. At most max_depth + 1 nodes are reported: a
 * deeper accepted path is cut to its first max_depth + 1 nodes. Unused
 * path slots hold -1. A malformed tree gives accept_len 0 and an all -1
 * path. argmax_out (may be NULL) gets -1 on padded rows and on every row
 * of a sequence whose n_nodes is out of range.
 */
void oracle_tree_verify(const uint16_t *logits, const int32_t *tokens, const int32_t *parents,
                        const int32_t *n_nodes, int32_t B, int32_t Nmax, int64_t V,
                        int32_t max_depth, int32_t *accept_len, int32_t *accept_path,
                        int32_t *argmax_out)
{
    int32_t *am = (int32_t *)malloc(sizeof(int32_t) * (size_t)Nmax);
    int32_t *chain = (int32_t *)malloc(sizeof(int32_t) * (size_t)Nmax);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *par = parents + (int64_t)b * Nmax;
        const int32_t *tok = tokens + (int64_t)b * Nmax;
        int32_t n = n_nodes[b];
        int n_ok = n >= 1 && n <= Nmax;
        for (int32_t i = 0; i < Nmax; ++i) am[i] = -1;
        if (n_ok) oracle_argmax_rows(logits + (int64_t)b * Nmax * V, n, V, am);
        if (argmax_out)
            for (int32_t i = 0; i < Nmax; ++i) argmax_out[(int64_t)b * Nmax + i] = am[i];
        int32_t *path = accept_path + (int64_t)b * (max_depth + 1);
        for (int32_t k = 0; k <= max_depth; ++k) path[k] = -1;
        if (!oracle_tree_is_valid(par, n, Nmax)) {
            accept_len[b] = 0;
            continue;
        }
        int32_t best = 0, best_depth = 0;
        accept_from(0, 0, par, tok, am, n, &best, &best_depth);
        int32_t len = ancestor_chain(par, best, chain);
        if (len > max_depth + 1) len = max_depth + 1;
        for (int32_t k = 0; k < len; ++k) path[k] = chain[k];
        accept_len[b] = len;
    }
    free(am);
    free(chain);
}

/*
 * Accepted-path KV commit ([paper] section 2.1: the prefix that the target
 * accepts extends the context). The accepted nodes' keys and values, taken
 * from the tree's own rows, become the next rows of the sequence's cache,
 * root first, and the prefix length grows by the number of nodes.
 *
 * For sequence b, with a = accept_len[b], P = prefix_lens[b], n = n_nodes[b]:
 *  - a == 0 (a malformed tree, as the verification reports it): nothing
 *    changes and flags[b] = 0;
 *  - the request is malformed if n is outside [1, Nmax], a outside
 *    [0, max_depth + 1] or above n (a path of tree nodes is no longer than
 *    the tree), P outside [0, Pcap], or a path entry path[b][k] (k < a)
 *    outside [0, n): nothing changes and flags[b] = 1;
 *  - the cache lacks room if P + a > Pcap: nothing changes and flags[b] = 2;
 *  - otherwise, for k < a and every kv head h, row P + k of head h of
 *    k_cache (v_cache) becomes tree_k[b][path[b][k]][h] (tree_v), bit for
 *    bit, prefix_lens[b] becomes P + a, and flags[b] = 0.
 * Layouts: tree_k/tree_v [B, Nmax, Hkv, d], k_cache/v_cache [B, Hkv, Pcap, d]
 * (bf16 bits), accept_path [B, max_depth + 1].
 */
void oracle_commit_kv(const uint16_t *tree_k, const uint16_t *tree_v, const int32_t *n_nodes,
                      const int32_t *accept_len, const int32_t *accept_path, uint16_t *k_cache,
                      uint16_t *v_cache, int32_t *prefix_lens, int32_t B, int32_t Nmax, int32_t Hkv,
                      int32_t d, int32_t Pcap, int32_t max_depth, int32_t *flags)
{
    for (int32_t b = 0; b < B; ++b) {
        const int32_t a = accept_len[b], P = prefix_lens[b], n = n_nodes[b];
        const int32_t *path = accept_path + (int64_t)b * (max_depth + 1);
        flags[b] = 0;
        if (a == 0) continue;
        int bad = n < 1 || n > Nmax || a < 0 || a > n || a > max_depth + 1 || P < 0 || P > Pcap;
        for (int32_t k = 0; !bad && k < a; ++k)
            if (path[k] < 0 || path[k] >= n) bad = 1;
        if (bad) {
            flags[b] = 1;
            continue;
        }
        if (P + a > Pcap) {
            flags[b] = 2;
            continue;
        }
        for (int32_t k = 0; k < a; ++k) {
            const int32_t node = path[k];
            for (int32_t h = 0; h < Hkv; ++h) {
                const int64_t src = (((int64_t)b * Nmax + node) * Hkv + h) * d;
                const int64_t dst = (((int64_t)b * Hkv + h) * Pcap + P + k) * d;
                for (int32_t e = 0; e < d; ++e) {
                    k_cache[dst + e] = tree_k[src + e];
                    v_cache[dst + e] = tree_v[src + e];
                }
            }
        }
        prefix_lens[b] = P + a;
    }
}

/*
 * Philox4x64-10, the counter-based generator of Salmon, Moraes, Dror and
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011): ten
 * rounds of two 64 x 64 -> 128-bit products on a 4-word counter, with the
 * 2-word key bumped by two Weyl constants after every round.
 */
void oracle_philox4x64_10(const uint64_t *ctr_in, const uint64_t *key, uint64_t *out)
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        const unsigned __int128 p0 = (unsigned __int128)M0 * c[0];
        const unsigned __int128 p1 = (unsigned __int128)M1 * c[2];
        const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
        k0 += W0;
        k1 += W1;
    }
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/*
 * The uniform number of stream `purpose` (0: acceptance tests, one per
 * node; 1: the Gumbel noise of the final sample, one per vocabulary entry)
 * for sequence b and item `index`: word index % 4 of the Philox block at
 * counter (index / 4, b, purpose, 0) under key (seed, offset), its top 23
 * bits as (k + 1/2) * 2^-23, strictly inside (0, 1).
 */
double oracle_uniform(uint64_t seed, uint64_t offset, uint32_t purpose, int32_t b, int64_t index)
{
    const uint64_t ctr[4] = {(uint64_t)index / 4, (uint64_t)(uint32_t)b, purpose, 0};
    const uint64_t key[2] = {seed, offset};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    const uint64_t w = out[index % 4];
    return ((double)(w >> 41) + 0.5) * ldexp(1.0, -23);
}

/* softmax(z / T) of one bf16 logits row, in double. */
static void softmax_row(const uint16_t *z, int64_t V, double T, double *p)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        const double x = bf16_to_double(z[v]) / T;
        if (x > m) m = x;
    }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        p[v] = exp(bf16_to_double(z[v]) / T - m);
        s += p[v];
    }
    for (int64_t v = 0; v < V; ++v) p[v] /= s;
}

/*
 * Stochastic tree verification at temperature T > 0: speculative sampling
 * ([paper] section 2.1 cites Leviathan et al. 2023 for the draft-then-verify
 * rule) applied at every accepted node to its children in index order.
 *
 * For sequence b, p_u = softmax(target[b][u] / T) is the target's
 * distribution after node u's path and q_u = softmax(draft[b][u] / T) the
 * draft's distribution from which u's children were drawn. Starting with
 * u = root and r = p_u, each child c of u (index order) with token x is
 * accepted iff U(c) < min(1, r(x) / q_u(x)), U(c) the acceptance uniform of
 * node c; on acceptance the walk moves to c with r = p_c. A rejected child
 * replaces r by the residual max(r - q_u, 0) / sum(max(r - q_u, 0)); if that
 * sum is 0 the remaining children are rejected and r = p_u. The walk also
 * stops at depth max_depth. The next token is then drawn from r by the
 * Gumbel-max rule: the v with r(v) > 0 maximising log r(v) + g(v),
 * g(v) = -log(-log U(v)) with U(v) the sampling uniform of entry v, the
 * lowest index on ties.
 *
 * Outputs: accept_len[b] (path nodes, root included), accept_path[b]
 * (root first, -1 padded), next_token[b]. A malformed tree gives 0, all -1
 * and -1. margins (may be NULL) gets per sequence the smallest
 * |U - min(1, ratio)| of the acceptance tests, the smallest residual mass,
 * and the gap between the two largest Gumbel keys, so that a test can tell
 * decisions that another precision could take differently (1 where none).
 */
void oracle_tree_verify_sample(const uint16_t *target, const uint16_t *draft, const int32_t *tokens,
                               const int32_t *parents, const int32_t *n_nodes, int32_t B, int32_t Nmax,
                               int64_t V, int32_t max_depth, double temperature, uint64_t seed,
                               uint64_t offset, int32_t *accept_len, int32_t *accept_path,
                               int32_t *next_token, double *margins)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *par = parents + (int64_t)b * Nmax;
        const int32_t *tok = tokens + (int64_t)b * Nmax;
        const int32_t n = n_nodes[b];
        int32_t *path = accept_path + (int64_t)b * (max_depth + 1);
        for (int32_t k = 0; k <= max_depth; ++k) path[k] = -1;
        double m_acc = 1.0, m_mass = 1.0, m_gap = 1.0;
        if (!oracle_tree_is_valid(par, n, Nmax)) {
            accept_len[b] = 0;
            next_token[b] = -1;
            if (margins) margins[3 * b] = margins[3 * b + 1] = margins[3 * b + 2] = 1.0;
            continue;
        }
        int32_t u = 0, depth = 0;
        path[0] = 0;
        for (;;) {
            const int64_t row = ((int64_t)b * Nmax + u) * V;
            softmax_row(target + row, V, temperature, p);
            for (int64_t v = 0; v < V; ++v) r[v] = p[v];
            int32_t next = -1;
            if (depth < max_depth) {
                softmax_row(draft + row, V, temperature, q);
                for (int32_t c = u + 1; c < n && next < 0; ++c) {
                    if (par[c] != u) continue;
                    const int32_t x = tok[c];
                    double ratio = (x >= 0 && x < V) ? (q[x] > 0.0 ? r[x] / q[x] : (r[x] > 0.0 ? 1.0 : 0.0)) : 0.0;
                    if (ratio > 1.0) ratio = 1.0;
                    const double U = oracle_uniform(seed, offset, 0, b, c);
                    if (fabs(U - ratio) < m_acc) m_acc = fabs(U - ratio);
                    if (U < ratio) {
                        next = c;
                        break;
                    }
                    double s = 0.0;
                    for (int64_t v = 0; v < V; ++v) {
                        r[v] = r[v] > q[v] ? r[v] - q[v] : 0.0;
                        s += r[v];
                    }
                    if (s < m_mass) m_mass = s;
                    if (!(s > 0.0)) {           /* the residual vanished */
                        for (int64_t v = 0; v < V; ++v) r[v] = p[v];
                        break;
                    }
                    for (int64_t v = 0; v < V; ++v) r[v] /= s;
                }
            }
            if (next < 0) break;
            u = next;
            path[++depth] = u;
        }
        double best = -INFINITY, second = -INFINITY;
        int32_t arg = -1;
        for (int64_t v = 0; v < V; ++v) {
            if (!(r[v] > 0.0)) continue;
            const double key = log(r[v]) - log(-log(oracle_uniform(seed, offset, 1, b, v)));
            if (key > best) {
                second = best;
                best = key;
                arg = (int32_t)v;
            } else if (key > second) {
                second = key;
            }
        }
        if (arg >= 0 && second > -INFINITY) m_gap = best - second;
        accept_len[b] = depth + 1;
        next_token[b] = arg;
        if (margins) {
            margins[3 * b] = m_acc;
            margins[3 * b + 1] = m_mass;
            margins[3 * b + 2] = m_gap;
        }
    }
    free(p);
    free(q);
    free(r);
}

/*
 * Draft-side path scoring. The blog's section "What JetFlow Does
 * Differently": the draft probability of a path is a product of
 * conditional distributions, each conditioned on the concrete ancestor
 * tokens of that branch.
 *
 * For sequence b, node u's row draft[b][u] holds the draft's logits for u's
 * children: log q_u(v) = z_v / T - log sum_w exp(z_w / T). Outputs:
 *  - node_lp[b][c] = log q_{parent(c)}(tokens[b][c]) for 0 < c < n, 0 for
 *    the root, -inf for a token outside [0, V); NaN on padding and on every
 *    node of a malformed tree;
 *  - path_lp[b][c] = the sum of node_lp over c's root path (the log of the
 *    product of conditionals), the same conventions;
 *  - with top_k > 0: the top_k most probable tokens of each node's row
 *    (larger logit first, the lower index on ties) and their log q_u,
 *    [B, Nmax, top_k] (-1 and NaN on padding / malformed);
 *  - with budget > 0: the expansion under a budget, the `budget` best
 *    candidates (u, v) among every node u < n and its top_k tokens v, by
 *    path score path_lp[u] + log q_u(v), larger first, ties to the lower
 *    (u, rank of v); [B, budget] parent node, token and score (-1, -1, NaN
 *    when fewer candidates exist or the tree is malformed).
 * Returns the smallest nonzero gap between consecutive candidate scores
 * in each sequence's selection and at its boundary in gaps[b] (may be
 * NULL), so that a test can tell orders another precision could make
 * differently (exactly equal scores come from equal logits of one row and
 * are ordered by rank in any precision).
 */
void oracle_tree_score(const uint16_t *draft, const int32_t *tokens, const int32_t *parents,
                       const int32_t *n_nodes, int32_t B, int32_t Nmax, int64_t V, double temperature,
                       int32_t top_k, int32_t budget, double *node_lp, double *path_lp, int32_t *topk_tok,
                       double *topk_lp, int32_t *cand_parent, int32_t *cand_token, double *cand_score,
                       double *gaps)
{
    double *lse = (double *)malloc(sizeof(double) * (size_t)Nmax);
    int32_t *chain = (int32_t *)malloc(sizeof(int32_t) * (size_t)Nmax);
    int64_t ncand_max = (int64_t)Nmax * (top_k > 0 ? top_k : 1);
    double *cs = (double *)malloc(sizeof(double) * (size_t)ncand_max);
    int32_t *cu = (int32_t *)malloc(sizeof(int32_t) * (size_t)ncand_max);
    int32_t *cj = (int32_t *)malloc(sizeof(int32_t) * (size_t)ncand_max);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *par = parents + (int64_t)b * Nmax;
        const int32_t *tok = tokens + (int64_t)b * Nmax;
        const int32_t n = n_nodes[b];
        const int ok = oracle_tree_is_valid(par, n, Nmax);
        for (int32_t i = 0; i < Nmax; ++i) {
            node_lp[(int64_t)b * Nmax + i] = NAN;
            path_lp[(int64_t)b * Nmax + i] = NAN;
            for (int32_t j = 0; j < top_k; ++j) {
                topk_tok[((int64_t)b * Nmax + i) * top_k + j] = -1;
                topk_lp[((int64_t)b * Nmax + i) * top_k + j] = NAN;
            }
        }
        for (int32_t j = 0; j < budget; ++j) {
            cand_parent[(int64_t)b * budget + j] = -1;
            cand_token[(int64_t)b * budget + j] = -1;
            cand_score[(int64_t)b * budget + j] = NAN;
        }
        if (gaps) gaps[b] = INFINITY;
        if (!ok) continue;
        for (int32_t u = 0; u < n; ++u) {
            const uint16_t *z = draft + ((int64_t)b * Nmax + u) * V;
            double m = -INFINITY, s = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                const double x = bf16_to_double(z[v]) / temperature;
                if (x > m) m = x;
            }
            for (int64_t v = 0; v < V; ++v) s += exp(bf16_to_double(z[v]) / temperature - m);
            lse[u] = m + log(s);
        }
        for (int32_t c = 0; c < n; ++c) {
            double lp = 0.0;
            if (c > 0) {
                const int32_t x = tok[c];
                lp = (x >= 0 && x < V)
                         ? bf16_to_double(draft[((int64_t)b * Nmax + par[c]) * V + x]) / temperature - lse[par[c]]
                         : -INFINITY;
            }
            node_lp[(int64_t)b * Nmax + c] = lp;
        }
        for (int32_t c = 0; c < n; ++c) {          /* the product of conditionals along the root path */
            const int32_t len = ancestor_chain(par, c, chain);
            double sum = 0.0;
            for (int32_t k = 0; k < len; ++k) sum += node_lp[(int64_t)b * Nmax + chain[k]];
            path_lp[(int64_t)b * Nmax + c] = sum;
        }
        /* top_k of each row: a list kept sorted while the row is read in
         * index order; an entry moves ahead only of strictly smaller ones,
         * so among equal logits the lower index stays first */
        for (int32_t u = 0; u < n && top_k > 0; ++u) {
            const uint16_t *z = draft + ((int64_t)b * Nmax + u) * V;
            int32_t *lt = topk_tok + ((int64_t)b * Nmax + u) * top_k;
            double *lv = topk_lp + ((int64_t)b * Nmax + u) * top_k;   /* holds logits until the end */
            int32_t cnt = 0;
            for (int64_t v = 0; v < V; ++v) {
                const double x = bf16_to_double(z[v]);
                if (cnt == top_k && !(x > lv[top_k - 1])) continue;
                int32_t pos = cnt < top_k ? cnt : top_k - 1;
                while (pos > 0 && x > lv[pos - 1]) {
                    lv[pos] = lv[pos - 1];
                    lt[pos] = lt[pos - 1];
                    --pos;
                }
                lv[pos] = x;
                lt[pos] = (int32_t)v;
                if (cnt < top_k) ++cnt;
            }
            for (int32_t j = 0; j < cnt; ++j) lv[j] = lv[j] / temperature - lse[u];
        }
        if (budget > 0 && top_k > 0) {
            int64_t nc = 0;
            for (int32_t u = 0; u < n; ++u)
                for (int32_t j = 0; j < top_k; ++j) {
                    if (topk_tok[((int64_t)b * Nmax + u) * top_k + j] < 0) continue;
                    cs[nc] = path_lp[(int64_t)b * Nmax + u] + topk_lp[((int64_t)b * Nmax + u) * top_k + j];
                    cu[nc] = u;
                    cj[nc] = j;
                    ++nc;
                }
            /* selection: take the best remaining candidate `budget` times */
            char *used = (char *)calloc((size_t)(nc > 0 ? nc : 1), 1);
            double prev = INFINITY;
            for (int32_t r = 0; r < budget && r < nc; ++r) {
                int64_t best = -1;
                for (int64_t k = 0; k < nc; ++k) {
                    if (used[k]) continue;
                    if (best < 0 || cs[k] > cs[best]) best = k;   /* ties: the earlier (u, j) */
                }
                used[best] = 1;
                cand_parent[(int64_t)b * budget + r] = cu[best];
                cand_token[(int64_t)b * budget + r] = topk_tok[((int64_t)b * Nmax + cu[best]) * top_k + cj[best]];
                cand_score[(int64_t)b * budget + r] = cs[best];
                if (gaps && r > 0 && prev - cs[best] > 0.0 && prev - cs[best] < gaps[b]) gaps[b] = prev - cs[best];
                prev = cs[best];
            }
            if (gaps && budget < nc) {               /* the boundary: the best candidate left out */
                double out = -INFINITY;
                for (int64_t k = 0; k < nc; ++k)
                    if (!used[k] && cs[k] > out) out = cs[k];
                if (prev - out > 0.0 && prev - out < gaps[b]) gaps[b] = prev - out;
            }
            free(used);
        }
    }
    free(lse);
    free(chain);
    free(cs);
    free(cu);
    free(cj);
}

/*
 * The accepted-path KV commit into a paged cache: the same request as
 * oracle_commit_kv, with row p of sequence b, head h stored at
 * k_pages[block_table[b][p / page_size]][p % page_size][h] (v_pages alike),
 * pages [num_pages, page_size, Hkv, d], block_table [B, pages_per_seq], the
 * capacity pages_per_seq * page_size. A request is also malformed (flags 1)
 * if a page holding one of rows P .. P + a - 1 is outside [0, num_pages).
 */
void oracle_commit_kv_paged(const uint16_t *tree_k, const uint16_t *tree_v, const int32_t *n_nodes,
                            const int32_t *accept_len, const int32_t *accept_path, uint16_t *k_pages,
                            uint16_t *v_pages, const int32_t *block_table, int32_t page_size, int32_t num_pages,
                            int32_t pages_per_seq, int32_t *prefix_lens, int32_t B, int32_t Nmax, int32_t Hkv,
                            int32_t d, int32_t max_depth, int32_t *flags)
{
    const int32_t Pcap = pages_per_seq * page_size;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t a = accept_len[b], P = prefix_lens[b], n = n_nodes[b];
        const int32_t *path = accept_path + (int64_t)b * (max_depth + 1);
        const int32_t *table = block_table + (int64_t)b * pages_per_seq;
        flags[b] = 0;
        if (a == 0) continue;
        int bad = n < 1 || n > Nmax || a < 0 || a > n || a > max_depth + 1 || P < 0 || P > Pcap;
        for (int32_t k = 0; !bad && k < a; ++k)
            if (path[k] < 0 || path[k] >= n) bad = 1;
        if (!bad && P + a <= Pcap)
            for (int32_t k = 0; k < a; ++k) {
                const int32_t ph = table[(P + k) / page_size];
                if (ph < 0 || ph >= num_pages) bad = 1;
            }
        if (bad) {
            flags[b] = 1;
            continue;
        }
        if (P + a > Pcap) {
            flags[b] = 2;
            continue;
        }
        for (int32_t k = 0; k < a; ++k) {
            const int32_t row = P + k, node = path[k];
            const int64_t page = table[row / page_size];
            for (int32_t h = 0; h < Hkv; ++h) {
                const int64_t src = (((int64_t)b * Nmax + node) * Hkv + h) * d;
                const int64_t dst = ((page * page_size + row % page_size) * Hkv + h) * d;
                for (int32_t e = 0; e < d; ++e) {
                    k_pages[dst + e] = tree_k[src + e];
                    v_pages[dst + e] = tree_v[src + e];
                }
            }
        }
        prefix_lens[b] = P + a;
    }
}
