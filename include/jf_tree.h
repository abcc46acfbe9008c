/*
 * jf_tree.h - C ABI of the GB300 (sm_103a) tree-attention and greedy
 * tree-verification library (libjf_tree.so).
 *
 * The method (JetFlow, arXiv 2606.18394; JetSpec on some pages) drafts a
 * tree of candidate tokens under the accepted prefix. The target model
 * verifies the whole tree in one parallel forward pass, then greedily
 * accepts the longest root path that its own predictions agree with.
 * This library provides the data-parallel hot path of that pass:
 *
 *   jf_tree_attention  one forward pass of tree-causal attention over the
 *                      whole tree ("JetFlow: Scaling Speculative Decoding
 *                      with Parallel Tree Drafting", blog, section "What
 *                      JetFlow Does Differently": every node attends to the
 *                      original prefix and to its own ancestors, never to
 *                      siblings or descendants; all nodes are computed in
 *                      one pass).
 *   jf_tree_verify     per-node vocabulary argmax, then the longest
 *                      accepted root path (the paper's section 2.1
 *                      "Background": the target verifies the N drafted
 *                      tokens in parallel and accepts the longest prefix
 *                      that agrees with its own predictions).
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is a CUDA device pointer on the current device.
 *    The caller owns every buffer, the workspace and the stream.
 *  - bf16 is IEEE bfloat16 (__nv_bfloat16) passed as raw 16-bit values.
 *  - Tensors are dense and row-major, in the layouts stated per argument.
 *  - Calls are asynchronous and ordered on `stream`, and they allocate no
 *    device memory. The return value reports only problems the host can
 *    see. Problems found on the device are OR-ed into `*status` (a device
 *    int32, may be NULL), which the caller reads after synchronising.
 *    The caller must zero it before the first call.
 *  - One workspace may serve a jf_tree_attention call and a jf_tree_verify
 *    call at the same time (the two use disjoint regions), but not two
 *    calls of the same entry point that overlap on the GPU.
 *
 * Tree encoding: parents[b][i] is the parent of node i of sequence b.
 * parents[b][0] = -1 (the root, i.e. the last committed token), and
 * 0 <= parents[b][i] < i for 0 < i < n_nodes[b] (topological order). Nodes
 * i >= n_nodes[b] are padding: they are neither read as tree nodes nor
 * written.
 */
#ifndef JF_TREE_H
#define JF_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define JF_API __attribute__((visibility("default")))
#else
#define JF_API
#endif

/* Opaque CUDA handles (cudaStream_t / cudaEvent_t). */
typedef struct CUstream_st *jf_stream_t;
typedef struct CUevent_st *jf_event_t;

/* Host return codes. */
enum {
    JF_OK = 0,
    JF_ERR_NULL = 1,      /* a required pointer is NULL */
    JF_ERR_SHAPE = 2,     /* a size is out of the supported range (see jf_shape) */
    JF_ERR_ALIGN = 3,     /* a tensor pointer is not 16-byte aligned */
    JF_ERR_WORKSPACE = 4, /* workspace_bytes < jf_workspace_bytes(shape) */
    JF_ERR_CUDA = 5       /* a CUDA runtime/driver call or kernel launch failed */
};

/* Device status flags, OR-ed into *status. */
enum {
    JF_STATUS_BAD_TREE = 1,  /* a sequence had n_nodes outside [1, max_nodes], a
                                parent breaking the encoding above, or (for
                                attention) prefix_lens outside [0, prefix_cap] */
    JF_STATUS_TIMEOUT = 2,   /* a kernel's bounded wait expired; outputs of the
                                call are undefined (never expected) */
    JF_STATUS_CACHE_FULL = 4 /* jf_tree_commit_kv: a sequence's accepted path
                                did not fit in its KV cache; that sequence
                                was left unchanged */
};

/*
 * Problem sizes.
 *   batch       B >= 1 sequences
 *   n_q_heads   Hq; n_kv_heads Hkv; Hq % Hkv == 0 and G = Hq / Hkv must be a
 *               power of two <= 128. Query head h reads KV head h / G.
 *   head_dim    d, 64 or 128
 *   max_nodes   Nmax, 1..256 tree slots per sequence
 *   prefix_cap  Pcap >= 1 rows per (sequence, KV head) in the KV cache
 *   vocab       V >= 1 and a multiple of 8 (jf_tree_verify only)
 *   scale       softmax scale; 0 selects 1/sqrt(d)
 */
typedef struct {
    int32_t batch;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t max_nodes;
    int32_t prefix_cap;
    int32_t vocab;
    float scale;
} jf_shape;

/*
 * Bytes of workspace that jf_tree_attention and jf_tree_verify need for
 * `shape` (one buffer serves both). Host-only, and needs no GPU. Returns 0
 * when the shape is outside the supported range. The size does not depend
 * on the prefix lengths or the trees, only on the shape.
 */
JF_API size_t jf_workspace_bytes(const jf_shape *shape);

/*
 * Tree-causal attention: one forward pass over every node of every tree.
 *
 * For node i of sequence b and query head h, with G = Hq / Hkv and kv = h / G:
 *   out[b,i,h,:] = softmax_j(scale * q[b,i,h,:] . K_j) V_j
 * over the keys j of the ordinary causal sequence that ends at node i:
 * the prefix rows k_cache[b,kv,0 .. prefix_lens[b]) followed by the tree
 * rows tree_k[b,a,kv,:] of every ancestor a of i and of i itself (the blog's
 * "What JetFlow Does Differently": each node attends to the prefix and to
 * its ancestors, never to siblings or descendants). V_j is the matching row
 * of v_cache / tree_v. RoPE and positions are the caller's: q and tree_k
 * arrive already rotated.
 *
 *   q            bf16 [B, Nmax, Hq, d]
 *   k_cache      bf16 [B, Hkv, Pcap, d]; rows >= prefix_lens[b] are never
 *   v_cache      bf16 [B, Hkv, Pcap, d]  used and may hold anything (NaN too)
 *   prefix_lens  int32 [B], each in [0, Pcap]
 *   tree_k       bf16 [B, Nmax, Hkv, d]; rows of padding nodes may hold anything
 *   tree_v       bf16 [B, Nmax, Hkv, d]
 *   parents      int32 [B, Nmax] (encoding above)
 *   n_nodes      int32 [B], each in [1, Nmax]
 *   out          bf16 [B, Nmax, Hq, d]; rows of padding nodes are not
 *                written; every row of a sequence flagged BAD_TREE is
 *                filled with NaN
 *   workspace    device buffer of >= jf_workspace_bytes(shape) bytes,
 *                256-byte aligned; its contents need no initialisation
 *   status       device int32 or NULL
 * Every bf16 pointer must be 16-byte aligned.
 * Repeat calls on one device give bit-identical results. The order in which
 * a row's keys are summed follows the work split over the SMs (and, when
 * the prefix keys and values of the call exceed half the L2, a rotated
 * order of the prefix tiles), so a device with another SM count may differ
 * in the last bits.
 * Returns JF_OK, JF_ERR_NULL, JF_ERR_SHAPE, JF_ERR_ALIGN, JF_ERR_WORKSPACE
 * or JF_ERR_CUDA.
 */
JF_API int32_t jf_tree_attention(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *prefix_lens, const void *tree_k,
                                 const void *tree_v, const int32_t *parents,
                                 const int32_t *n_nodes, void *out, const jf_shape *shape,
                                 void *workspace, size_t workspace_bytes, int32_t *status,
                                 jf_stream_t stream);

/*
 * Tree attention over a paged prefix cache: jf_tree_attention with the
 * prefix keys and values in fixed-size pages reached through a block table
 * (the cache layout of paged serving engines), so that sequences share one
 * page pool. Row p of sequence b's prefix, KV head h, is
 *   k_pages[block_table[b, p / page_size], p % page_size, h, :]
 * (v_pages alike). Everything else is as for jf_tree_attention.
 *
 *   k_pages, v_pages bf16 [num_pages, page_size, Hkv, d]
 *   block_table      int32 [B, prefix_cap / page_size]; entries for pages
 *                    past ceil(prefix_lens[b] / page_size) are never read
 *   page_size        a power of two from 8 to 128 dividing shape->prefix_cap
 *                    (else JF_ERR_SHAPE)
 *   num_pages        pages in the pool, >= 1
 * A used block-table entry outside [0, num_pages) makes the sequence
 * malformed: NaN rows and JF_STATUS_BAD_TREE.
 */
JF_API int32_t jf_tree_attention_paged(const void *q, const void *k_pages, const void *v_pages,
                                       const int32_t *block_table, int32_t page_size, int32_t num_pages,
                                       const int32_t *prefix_lens, const void *tree_k,
                                       const void *tree_v, const int32_t *parents,
                                       const int32_t *n_nodes, void *out, const jf_shape *shape,
                                       void *workspace, size_t workspace_bytes, int32_t *status,
                                       jf_stream_t stream);

/*
 * Greedy tree verification.
 *
 * am[b,i] = argmax_v logits[b,i,v] for i < n_nodes[b], the lowest index on
 * ties, +0 == -0, and a NaN ranks above every number (the first NaN wins).
 * A non-root node c is accepted iff its parent p is accepted and
 * tree_tokens[b,c] == am[b,p]; the root is always accepted (its token is
 * not checked). The reported node is the deepest accepted node (lowest
 * index on ties). Its root path, root first, goes to accept_path_out,
 * and accept_len_out counts that path's nodes, root included (the paper's
 * section 2.1 "Background": accept the longest prefix that agrees with the
 * target's predictions). Only max_depth + 1 path slots exist, so a deeper
 * accepted path is cut to its first max_depth + 1 nodes. The bonus token
 * of greedy decoding is am at the last reported node (in argmax_out).
 *
 *   logits           bf16 [B, Nmax, V], 16-byte aligned
 *   tree_tokens      int32 [B, Nmax]
 *   parents, n_nodes as for jf_tree_attention
 *   accept_len_out   int32 [B]; 0 for a sequence flagged BAD_TREE
 *   accept_path_out  int32 [B, max_depth + 1]; unused slots -1
 *   argmax_out       int32 [B, Nmax] or NULL; -1 on padding rows and on
 *                    every row of a sequence whose n_nodes is out of range
 *   max_depth        >= 0
 * Returns as jf_tree_attention.
 */
JF_API int32_t jf_tree_verify(const void *logits, const int32_t *tree_tokens,
                              const int32_t *parents, const int32_t *n_nodes,
                              int32_t *accept_len_out, int32_t *accept_path_out,
                              int32_t *argmax_out, const jf_shape *shape, int32_t max_depth,
                              void *workspace, size_t workspace_bytes, int32_t *status,
                              jf_stream_t stream);

/*
 * Stochastic tree verification at temperature T > 0: speculative sampling
 * (the paper's section 2.1 "Background" cites Leviathan et al. 2023 for the
 * draft-then-verify rule) applied along the tree.
 *
 * For sequence b, p_u = softmax(target_logits[b, u] / T) is the target's
 * distribution after node u's path and q_u = softmax(draft_logits[b, u] / T)
 * the draft's distribution from which u's children were drawn. From the
 * root, with r = p_u, each child c of the current node u (index order)
 * with token x = tree_tokens[b, c] is accepted iff U(c) < min(1, r(x) /
 * q_u(x)); the walk then moves to c with r = p_c. A rejected child replaces
 * r by max(r - q_u, 0) renormalised; if that residual is 0 everywhere the
 * remaining children are rejected and r = p_u. The walk stops at a node
 * with no accepted child or at depth max_depth, and next_token_out[b] is
 * drawn from r by the Gumbel-max rule: the v with r(v) > 0 maximising
 * ln r(v) - ln(-ln U'(v)), the lowest index on ties. A token outside
 * [0, V) is always rejected.
 *
 * Random numbers: Philox4x64-10 (Salmon et al., "Parallel random numbers:
 * as easy as 1, 2, 3", SC 2011) under the key (seed, offset). U(c) is word
 * c % 4 of the block at counter (c / 4, b, 0, 0); U'(v) is word v % 4 of
 * the block at counter (v / 4, b, 1, 0); a word w gives the uniform
 * (floor(w / 2^41) + 1/2) / 2^23. Pass a new offset (e.g. the decoding
 * step) for fresh numbers. The arithmetic is fp32 (normalisers from
 * chunked sums), so a decision whose margin is within rounding of fp32
 * may differ from an exact evaluation.
 *
 *   target_logits, draft_logits  bf16 [B, Nmax, V], finite values
 *   tree_tokens, parents, n_nodes as for jf_tree_verify
 *   temperature      > 0 and finite, else JF_ERR_SHAPE
 *   seed, offset     the Philox key
 *   accept_len_out   int32 [B]: path nodes including the root (>= 1),
 *                    0 for a malformed tree
 *   accept_path_out  int32 [B, max_depth + 1], root first, -1 padded
 *   next_token_out   int32 [B]: the token sampled after the path, -1 for a
 *                    malformed tree
 *   max_depth        >= 0: the walk goes no deeper
 * The workspace is the one jf_workspace_bytes(shape) sizes. Each sequence
 * is walked by a cluster of 16 CTAs (8 when B * 16 exceeds the SM count or
 * the device refuses clusters of 16). Returns as jf_tree_verify; a
 * malformed tree raises JF_STATUS_BAD_TREE.
 */
JF_API int32_t jf_tree_verify_sample(const void *target_logits, const void *draft_logits,
                                     const int32_t *tree_tokens, const int32_t *parents,
                                     const int32_t *n_nodes, float temperature, uint64_t seed,
                                     uint64_t offset, int32_t *accept_len_out,
                                     int32_t *accept_path_out, int32_t *next_token_out,
                                     const jf_shape *shape, int32_t max_depth, void *workspace,
                                     size_t workspace_bytes, int32_t *status, jf_stream_t stream);

/*
 * Draft-side path scoring: the step before verification. The blog's
 * section "What JetFlow Does Differently": a path's draft probability is
 * the product of conditional distributions, each on the concrete ancestor
 * tokens of its branch. Row u of draft_logits holds the draft's logits for
 * node u's children: log q_u(v) = z_v / T - log sum_w exp(z_w / T).
 *
 *   draft_logits     bf16 [B, Nmax, V], finite values
 *   tree_tokens, parents, n_nodes as for jf_tree_verify
 *   temperature      > 0 and finite
 *   top_k            0..16: how many of each row's most probable tokens to
 *                    report (the larger logit first, the lower index on ties)
 *   budget           0..Nmax * top_k (0 when top_k = 0): how many expansion
 *                    candidates to select
 *   node_logprob_out float32 [B, Nmax]: log q_{parent(c)}(tree_tokens[c]),
 *                    0 for the root, -inf for a token outside [0, V)
 *   path_logprob_out float32 [B, Nmax]: the sum of node_logprob over the
 *                    node's root path (the log of the path's probability)
 *   topk_token_out   int32 [B, Nmax, top_k] (NULL when top_k = 0)
 *   topk_logprob_out float32 [B, Nmax, top_k]: log q_u of those tokens
 *   cand_parent_out, cand_token_out int32 [B, budget], cand_score_out
 *                    float32 [B, budget] (NULL when budget = 0): the
 *                    `budget` best candidates (u, v) among every node u and
 *                    its top_k tokens, by path score path_logprob[u] +
 *                    log q_u(v), larger first, ties to the lower (u, rank)
 * Padding nodes and every node of a malformed tree get NaN (-1 for the
 * integers), and a malformed tree raises JF_STATUS_BAD_TREE. The
 * arithmetic is fp32; the selection orders by fp32 scores. The workspace
 * is the one jf_workspace_bytes(shape) sizes. Returns as jf_tree_verify.
 */
JF_API int32_t jf_tree_score(const void *draft_logits, const int32_t *tree_tokens,
                             const int32_t *parents, const int32_t *n_nodes, float temperature,
                             int32_t top_k, int32_t budget, float *node_logprob_out,
                             float *path_logprob_out, int32_t *topk_token_out,
                             float *topk_logprob_out, int32_t *cand_parent_out,
                             int32_t *cand_token_out, float *cand_score_out,
                             const jf_shape *shape, void *workspace, size_t workspace_bytes,
                             int32_t *status, jf_stream_t stream);

/*
 * Accepted-path KV commit: the step after verification (the paper's section
 * 2.1 "Background": the prefix the target accepts extends the context). The
 * keys and values of the accepted nodes were computed by this tree's
 * attention pass (tree_k / tree_v rows); they become the next rows of each
 * sequence's KV cache, root first, and the prefix length grows by the
 * number of nodes.
 *
 * For sequence b, with a = accept_len[b] and P = prefix_lens[b]: for k < a
 * and every kv head h, row P + k of head h of k_cache becomes
 * tree_k[b, accept_path[b, k], h, :] (v_cache from tree_v alike), bit for
 * bit, and prefix_lens[b] becomes P + a. With a = 0 (what jf_tree_verify
 * reports for a malformed tree) nothing changes.
 *
 *   tree_k, tree_v   bf16 [B, Nmax, Hkv, d], as for jf_tree_attention
 *   n_nodes          int32 [B]
 *   accept_len       int32 [B]           (from jf_tree_verify)
 *   accept_path      int32 [B, max_depth + 1]  (from jf_tree_verify)
 *   k_cache, v_cache bf16 [B, Hkv, Pcap, d], updated in place
 *   prefix_lens      int32 [B], updated in place (the same array the next
 *                    jf_tree_attention call reads)
 *   shape, max_depth as for jf_tree_attention / jf_tree_verify
 *   status           device int32 or NULL
 * A sequence whose request is malformed (n_nodes outside [1, Nmax],
 * accept_len outside [0, min(n_nodes, max_depth + 1)], prefix_lens outside
 * [0, Pcap], or a path entry that is not a node of the tree) raises
 * JF_STATUS_BAD_TREE; one whose path does not fit (P + a > Pcap) raises
 * JF_STATUS_CACHE_FULL. Either way that sequence is left unchanged.
 * Every bf16 pointer must be 16-byte aligned. The call needs no workspace
 * and allocates nothing.
 * Returns JF_OK, JF_ERR_NULL, JF_ERR_SHAPE, JF_ERR_ALIGN or JF_ERR_CUDA.
 */
JF_API int32_t jf_tree_commit_kv(const void *tree_k, const void *tree_v, const int32_t *n_nodes,
                                 const int32_t *accept_len, const int32_t *accept_path, void *k_cache,
                                 void *v_cache, int32_t *prefix_lens, const jf_shape *shape,
                                 int32_t max_depth, int32_t *status, jf_stream_t stream);

/*
 * The accepted-path KV commit into a paged cache (the pool and block table
 * of jf_tree_attention_paged): jf_tree_commit_kv with row p of sequence b
 * stored at k_pages[block_table[b, p / page_size], p % page_size, h, :]
 * (v_pages alike). The pages that receive rows P .. P + a - 1 must already
 * be in the sequence's block table; a request is also malformed
 * (JF_STATUS_BAD_TREE, nothing changes) if one of them lies outside
 * [0, num_pages). The capacity is shape->prefix_cap (= block-table width x
 * page_size); page_size and num_pages as for jf_tree_attention_paged.
 */
JF_API int32_t jf_tree_commit_kv_paged(const void *tree_k, const void *tree_v,
                                       const int32_t *n_nodes, const int32_t *accept_len,
                                       const int32_t *accept_path, void *k_pages, void *v_pages,
                                       const int32_t *block_table, int32_t page_size,
                                       int32_t num_pages, int32_t *prefix_lens,
                                       const jf_shape *shape, int32_t max_depth, int32_t *status,
                                       jf_stream_t stream);

/*
 * Allocation-free variant of jf_tree_verify. The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory.
 * Examples: code running inside a CUDA graph capture, a custom allocator
 * that owns all of the device's memory, or an embedding that forbids
 * cudaMalloc after start-up. Such callers cannot provide a workspace.
 *
 * It computes exactly what jf_tree_verify computes, with the same arguments
 * minus the workspace. Its scratch (the per-chunk argmax partials) is a
 * fixed array of JF_NOALLOC_SCRATCH_BYTES in the library's device memory.
 * Every GPU that loads the library holds that array until the process
 * exits. The call itself allocates nothing.
 *  - Limit: rows * chunks * 8 bytes must be <= JF_NOALLOC_SCRATCH_BYTES,
 *    with rows = batch * max_nodes and chunks the argmax pieces per logits
 *    row, at most max(ceil(vocab / 76800), ceil(4 * SMs / rows)) (608 / rows
 *    on a 152-SM GB300). For vocab 151936 that is 2 from 304 rows up, so
 *    every problem that the row limit of jf_tree_verify admits (at most 65535
 *    rows) fits. Larger problems return JF_ERR_SHAPE and launch nothing.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it with the device's current context;
 *    a call under another context (after cudaDeviceReset, for example)
 *    looks it up again. Make the first call on a context before any stream
 *    capture.
 *  - All calls share the one array, and each call overwrites what it
 *    reads. Calls that overlap on the GPU (on different streams, or on
 *    different host threads without ordering) race on it, so serialise
 *    them.
 * Returns as jf_tree_verify; JF_ERR_CUDA if the address lookup fails.
 */
#define JF_NOALLOC_SCRATCH_BYTES (1u << 20)
JF_API int32_t jf_tree_verify_noalloc(const void *logits, const int32_t *tree_tokens,
                                      const int32_t *parents, const int32_t *n_nodes,
                                      int32_t *accept_len_out, int32_t *accept_path_out,
                                      int32_t *argmax_out, const jf_shape *shape,
                                      int32_t max_depth, int32_t *status, jf_stream_t stream);

/* Static description of a return code or status flag. */
JF_API const char *jf_status_string(int32_t code);

/*
 * Instrumentation (host-only bookkeeping; adds no device work).
 *
 * jf_kernel_launch_count: kernels this library has launched in this process.
 *
 * jf_trace_kernels: arm per-kernel timing. `events` holds 2 * capacity
 * cudaEvent_t handles created by the caller with timing enabled. Each
 * following kernel launch records events[2k] before and events[2k+1] after
 * itself on the launch stream, for k = 0, 1, ... < capacity. A call with
 * capacity 0 (or events NULL) disarms. The caller keeps `events` alive while
 * armed.
 * jf_trace_count: pairs recorded since the last arm.
 * jf_trace_name: name of the kernel that recorded pair k (NULL if none).
 */
JF_API uint64_t jf_kernel_launch_count(void);
JF_API int32_t jf_trace_kernels(jf_event_t *events, int32_t capacity);
JF_API int32_t jf_trace_count(void);
JF_API const char *jf_trace_name(int32_t k);

#ifdef __cplusplus
}
#endif

#endif /* JF_TREE_H */
