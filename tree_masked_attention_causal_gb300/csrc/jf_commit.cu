// jf_commit.cu - accepted-path KV commit on sm_103a.
//
// The paper's section 2.1 "Background": the prefix the target accepts
// extends the context. After greedy verification the accepted path's nodes
// (root first) become the next rows of each sequence's KV cache: their keys
// and values are the tree's own rows, already computed by the attention pass
// with the right positions, so committing them is a copy, and the prefix
// length grows by the path length.
//
// The cache is contiguous ([B, Hkv, Pcap, d]) or paged ([num_pages,
// page_size, Hkv, d] through a block table, as jf_tree_attention_paged
// reads it).
//
// One block per sequence (so that reading and raising prefix_lens[b] cannot
// race with another block), 512 threads. The block checks the request, then
// copies a * Hkv key rows and as many value rows in 16-byte pieces: each
// thread loads up to four pieces before it stores any, so that the block
// waits for one round of memory latency per 2048 pieces instead of one per
// piece. The length is raised last.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kCommitThreads = 512;
constexpr int kCommitBatch = 4;          // pieces in flight per thread

__global__ void __launch_bounds__(kCommitThreads)
    commit_kv_kernel(const __nv_bfloat16 *__restrict__ tree_k, const __nv_bfloat16 *__restrict__ tree_v,
                     const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ accept_len,
                     const int32_t *__restrict__ accept_path, __nv_bfloat16 *__restrict__ k_cache,
                     __nv_bfloat16 *__restrict__ v_cache, int32_t *__restrict__ prefix_lens, int Nmax, int Hkv,
                     int D, int Pcap, int max_depth, int32_t *status, const int32_t *__restrict__ block_table,
                     int page_lg, int pages_per_seq, int num_pages) {
    // A programmatic dependent of the stream's previous kernel (normally the
    // accept walk): nothing is read before that grid has completed. A
    // follower may launch once this kernel has started.
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    __shared__ int s_node[kMaxNodes + 1];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int a = accept_len[b], P = prefix_lens[b], n = n_nodes[b];
    const int32_t *path = accept_path + (size_t)b * (max_depth + 1);
    if (a == 0) return;                                   // nothing accepted (a malformed tree)
    // The request: n in [1, Nmax], a in [0, min(n, max_depth + 1)] (a path of
    // tree nodes is no longer than the tree), P in [0, Pcap], every path
    // entry a node of the tree; then room for a more rows.
    bool bad = n < 1 || n > Nmax || a < 0 || a > n || a > max_depth + 1 || P < 0 || P > Pcap;
    for (int k = tid; !bad && k < a; k += kCommitThreads) {
        const int node = path[k];
        if (node < 0 || node >= n) bad = true;
        else s_node[k] = node;
    }
    bad = __syncthreads_or(bad);
    // paged: every page that receives a row must be a page of the pool
    if (!bad && page_lg >= 0 && P + a <= Pcap) {
        for (int k = tid; k < a; k += kCommitThreads) {
            const int ph = block_table[(size_t)b * pages_per_seq + ((P + k) >> page_lg)];
            if (ph < 0 || ph >= num_pages) bad = true;
        }
        bad = __syncthreads_or(bad);
    }
    if (bad || P + a > Pcap) {
        if (tid == 0) set_status(status, bad ? JF_STATUS_BAD_TREE : JF_STATUS_CACHE_FULL);
        return;
    }
    // a rows x Hkv heads x (K, V), d / 8 sixteen-byte pieces each: piece e
    // of row (k, h) of K (kv = 0) or V (kv = 1)
    const int pieces = D / 8;
    const int total = a * Hkv * 2 * pieces;
    auto locate = [&](int idx, const uint4 *&s, uint4 *&t) {
        const int e = idx % pieces;
        int r = idx / pieces;
        const int kv = r & 1;
        r >>= 1;
        const int h = r % Hkv, k = r / Hkv;
        const size_t src = (((size_t)b * Nmax + s_node[k]) * Hkv + h) * D + e * 8;
        size_t dst;
        if (page_lg < 0) {
            dst = (((size_t)b * Hkv + h) * Pcap + P + k) * D + e * 8;
        } else {                                      // [num_pages, page_size, Hkv, d]
            const int row = P + k;
            const size_t ph = (size_t)block_table[(size_t)b * pages_per_seq + (row >> page_lg)];
            dst = (((ph << page_lg) + (row & ((1 << page_lg) - 1))) * Hkv + h) * D + e * 8;
        }
        s = reinterpret_cast<const uint4 *>((kv ? tree_v : tree_k) + src);
        t = reinterpret_cast<uint4 *>((kv ? v_cache : k_cache) + dst);
    };
    for (int base = 0; base < total; base += kCommitThreads * kCommitBatch) {
        uint4 v[kCommitBatch];
        uint4 *to[kCommitBatch];
#pragma unroll
        for (int j = 0; j < kCommitBatch; ++j) {
            const int idx = base + j * kCommitThreads + tid;
            to[j] = nullptr;
            if (idx < total) {
                const uint4 *from;
                locate(idx, from, to[j]);
                v[j] = __ldg(from);
            }
        }
#pragma unroll
        for (int j = 0; j < kCommitBatch; ++j)
            if (to[j]) *to[j] = v[j];
    }
    __syncthreads();
    if (tid == 0) prefix_lens[b] = P + a;                 // last: every row is written
}

}  // namespace

cudaError_t launch_commit_kv(const Layout &L, const __nv_bfloat16 *tree_k, const __nv_bfloat16 *tree_v,
                             const int32_t *n_nodes, const int32_t *accept_len, const int32_t *accept_path,
                             __nv_bfloat16 *k_cache, __nv_bfloat16 *v_cache, int32_t *prefix_lens, int32_t max_depth,
                             int32_t *status, cudaStream_t s, const int32_t *block_table, int32_t page_lg,
                             int32_t num_pages) {
    trace_begin("commit_kv", s);
    const int pages_per_seq = page_lg >= 0 ? L.Pcap >> page_lg : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(L.B, 1, 1);
    cfg.blockDim = dim3(kCommitThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, commit_kv_kernel, tree_k, tree_v, n_nodes, accept_len, accept_path,
                                       k_cache, v_cache, prefix_lens, (int)L.Nmax, (int)L.Hkv, (int)L.D,
                                       (int)L.Pcap, (int)max_depth, status, block_table, (int)page_lg,
                                       pages_per_seq, (int)num_pages);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(s);
    return e;
}

}  // namespace jf
