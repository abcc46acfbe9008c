// jf_api.cu - the C ABI (include/jf_tree.h): argument validation, workspace
// layout, TMA tensor-map encoding and the stream-ordered kernel launches.
//
// Every check that needs no GPU runs before the first CUDA call, so bad
// arguments are reported (and testable) on a machine without a GPU.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "jf_common.cuh"

namespace jf {

// ------------------------------------------------------------- tracing
namespace {
std::atomic<uint64_t> g_launches{0};
std::mutex g_trace_mu;
jf_event_t *g_trace_events = nullptr;
int32_t g_trace_capacity = 0;
int32_t g_trace_count = 0;
const char *g_trace_names[4096];
thread_local bool t_open = false;

// Inside stream capture a plain event record is only a dependency marker;
// the external flag makes it a timing-capable event node of the graph.
void record(jf_event_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(reinterpret_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal);
    else
        cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), s);
}
}  // namespace

void trace_begin(const char *name, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(g_trace_mu);
    t_open = false;
    if (g_trace_events && g_trace_count < g_trace_capacity) {
        record(g_trace_events[2 * g_trace_count], s);
        if (g_trace_count < 4096) g_trace_names[g_trace_count] = name;
        t_open = true;
    }
}

void trace_end(cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (t_open && g_trace_events && g_trace_count < g_trace_capacity) {
        record(g_trace_events[2 * g_trace_count + 1], s);
        ++g_trace_count;
    }
    t_open = false;
}

// -------------------------------------------------------- validation
namespace {

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Shape checks shared by both entry points; `need_vocab` for verify.
int32_t check_shape(const jf_shape *s, bool need_vocab, bool need_attn) {
    if (!s) return JF_ERR_NULL;
    if (s->batch < 1 || s->max_nodes < 1 || s->max_nodes > kMaxNodes) return JF_ERR_SHAPE;
    if (need_attn) {
        if (s->n_q_heads < 1 || s->n_kv_heads < 1 || s->n_q_heads % s->n_kv_heads) return JF_ERR_SHAPE;
        const int G = s->n_q_heads / s->n_kv_heads;
        if (!pow2(G) || G > kBM) return JF_ERR_SHAPE;   // kRows / G >= 2 nodes per unit
        if (s->head_dim != 64 && s->head_dim != 128) return JF_ERR_SHAPE;
        if (s->prefix_cap < 1 || s->batch > kMaxBatch) return JF_ERR_SHAPE;
        if (!(s->scale >= 0.0f) || isinf(s->scale)) return JF_ERR_SHAPE;
        // 32-bit index arithmetic in the kernels
        if ((long long)s->batch * s->max_nodes * s->n_q_heads * s->head_dim > 0x7FFFFFFFll) return JF_ERR_SHAPE;
        if ((long long)s->batch * s->n_kv_heads * s->prefix_cap > 0x7FFFFFFFll) return JF_ERR_SHAPE;
        // the stream-K plan counts key tiles of all work units in 32 bits
        const long long units = (long long)s->batch * s->n_kv_heads * ((s->max_nodes * G + kRows - 1) / kRows);
        if (units * ((s->prefix_cap + kBN - 1) / kBN + (s->max_nodes + kBN - 1) / kBN + kSwitchTiles) > 0x7FFFFFFFll)
            return JF_ERR_SHAPE;
    }
    if (need_vocab) {
        if (s->vocab < 8 || s->vocab % 8) return JF_ERR_SHAPE;
        if ((long long)s->batch * s->max_nodes > 65535) return JF_ERR_SHAPE;   // grid.y
    }
    return JF_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Fully-defined shapes for the workspace: attention fields count only if
// they are valid, vocab only if it is valid. Both entry points and
// jf_workspace_bytes use this one layout, so their offsets always agree.
bool attn_shape_ok(const jf_shape *s) { return check_shape(s, false, true) == JF_OK; }
bool verify_shape_ok(const jf_shape *s) { return check_shape(s, true, false) == JF_OK; }

// `sms`: the device's SM count in a call, kMaxSms for jf_workspace_bytes.
Layout layout_of(const jf_shape *shape, int sms = kMaxSms) {
    jf_shape s = *shape;
    if (!attn_shape_ok(&s)) { s.n_q_heads = 1; s.n_kv_heads = 1; s.head_dim = 64; s.prefix_cap = 1; }
    if (!verify_shape_ok(&s)) s.vocab = 8;
    return make_layout(s.batch, s.max_nodes, s.n_q_heads, s.n_kv_heads, s.head_dim, s.prefix_cap, s.vocab,
                       sms < kMaxSms ? sms : kMaxSms);
}

// ----------------------------------------------------- device queries
int num_sms_cached(int dev) {
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = v;
    }
    return cache[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D 16-bit map, 128-byte swizzle, zero fill out of bounds. dims/box are
// innermost first; strides are the byte strides of dims 1 and 2.
bool encode3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
              uint32_t b0, uint32_t b1, uint32_t b2,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace jf

using namespace jf;

extern "C" {

JF_API size_t jf_workspace_bytes(const jf_shape *shape) {
    if (!shape || (!attn_shape_ok(shape) && !verify_shape_ok(shape))) return 0;
    return layout_of(shape).total;
}

JF_API const char *jf_status_string(int32_t code) {
    switch (code) {
        case JF_OK: return "ok";
        case JF_ERR_NULL: return "a required pointer is NULL";
        case JF_ERR_SHAPE: return "a size is outside the supported range";
        case JF_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
        case JF_ERR_WORKSPACE: return "workspace too small";
        case JF_ERR_CUDA: return "CUDA call or kernel launch failed";
        default: break;
    }
    return "unknown status code";
}

// The attention call over a contiguous cache (page_size 0) or a paged one.
static int32_t attention_call(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                              int32_t page_size, int32_t num_pages, const int32_t *prefix_lens, const void *tree_k,
                              const void *tree_v, const int32_t *parents, const int32_t *n_nodes, void *out,
                              const jf_shape *shape, void *workspace, size_t workspace_bytes, int32_t *status,
                              jf_stream_t stream) {
    if (!q || !k_cache || !v_cache || !prefix_lens || !tree_k || !tree_v || !parents || !n_nodes || !out || !shape ||
        !workspace || (page_size > 0 && !block_table))
        return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, false, true);
    if (sc != JF_OK) return sc;
    int page_lg = -1;
    if (page_size > 0) {
        page_lg = 0;
        while ((1 << page_lg) < page_size) ++page_lg;
        // a power of two from 8 to 128 (whole 1024-byte swizzle atoms, at most
        // one tile), a whole number of pages per sequence, and page rows
        // addressable in 32 bits
        if ((1 << page_lg) != page_size || page_size < 8 || page_size > kBN || shape->prefix_cap % page_size ||
            num_pages < 1 || (long long)num_pages * page_size > 0x7FFFFFFFll)
            return JF_ERR_SHAPE;
    }
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(tree_k) || !aligned16(tree_v) ||
        !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return JF_ERR_ALIGN;
    if (workspace_bytes < jf_workspace_bytes(shape)) return JF_ERR_WORKSPACE;

    const Layout L = layout_of(shape);
    const int B = shape->batch, N = shape->max_nodes, Hq = shape->n_q_heads, Hkv = shape->n_kv_heads;
    const int D = shape->head_dim, Pcap = shape->prefix_cap;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
    const int sms = num_sms_cached(dev);
    if (sms <= 0) return JF_ERR_CUDA;

    AttnMaps maps;
    const uint64_t e2 = 2;   // bytes per bf16
    bool ok = encode3d(&maps.q, q, D, Hq, (uint64_t)B * N, e2 * D, e2 * D * Hq, 64, L.G, L.NB);
    if (page_size > 0) {     // [num_pages, page_size, Hkv, d]: one box is one page of one head
        const uint64_t rows = (uint64_t)num_pages * page_size;
        ok = ok && encode3d(&maps.k_cache, k_cache, D, Hkv, rows, e2 * D, e2 * D * Hkv, 64, 1, page_size);
        ok = ok && encode3d(&maps.v_cache, v_cache, D, Hkv, rows, e2 * D, e2 * D * Hkv, 64, 1, page_size);
    } else {
        ok = ok && encode3d(&maps.k_cache, k_cache, D, Pcap, (uint64_t)B * Hkv, e2 * D, e2 * D * Pcap, 64, kBN, 1);
        ok = ok && encode3d(&maps.v_cache, v_cache, D, Pcap, (uint64_t)B * Hkv, e2 * D, e2 * D * Pcap, 64, kBN, 1);
    }
    ok = ok && encode3d(&maps.tree_k, tree_k, D, Hkv, (uint64_t)B * N, e2 * D, e2 * D * Hkv, 64, 1, kBN);
    ok = ok && encode3d(&maps.tree_v, tree_v, D, Hkv, (uint64_t)B * N, e2 * D, e2 * D * Hkv, 64, 1, kBN);
    ok = ok && encode3d(&maps.out, out, D, Hq, (uint64_t)B * N, e2 * D, e2 * D * Hq, 64, L.G, L.NB);
    ok = ok && encode3d(&maps.part, static_cast<uint8_t *>(workspace) + L.opart_off, D, kRows, L.max_pieces, e2 * D,
                        e2 * D * kRows, 64, kRows, 1, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    if (!ok) return JF_ERR_CUDA;

    AttnArgs args;
    args.prefix_lens = prefix_lens;
    args.parents = parents;
    args.n_nodes = n_nodes;
    args.out = reinterpret_cast<__nv_bfloat16 *>(out);
    args.ws = reinterpret_cast<uint8_t *>(workspace);
    args.status = status;
    const float scale = shape->scale > 0.f ? shape->scale : 1.0f / sqrtf((float)D);
    args.scale_log2 = scale * 1.4426950408889634f;
    args.num_ctas = sms < kMaxCtas ? sms : kMaxCtas;
    args.block_table = block_table;
    args.page_lg = page_lg;
    args.pages_per_seq = page_size > 0 ? Pcap / page_size : 0;
    args.num_pages = page_size > 0 ? num_pages : 0;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_tree_attention(L, maps, args, s) != cudaSuccess) return JF_ERR_CUDA;
    if (launch_split_combine(L, args, s) != cudaSuccess) return JF_ERR_CUDA;
    return JF_OK;
}

JF_API int32_t jf_tree_attention(const void *q, const void *k_cache, const void *v_cache, const int32_t *prefix_lens,
                                 const void *tree_k, const void *tree_v, const int32_t *parents,
                                 const int32_t *n_nodes, void *out, const jf_shape *shape, void *workspace,
                                 size_t workspace_bytes, int32_t *status, jf_stream_t stream) {
    return attention_call(q, k_cache, v_cache, nullptr, 0, 0, prefix_lens, tree_k, tree_v, parents, n_nodes, out,
                          shape, workspace, workspace_bytes, status, stream);
}

JF_API int32_t jf_tree_attention_paged(const void *q, const void *k_pages, const void *v_pages,
                                       const int32_t *block_table, int32_t page_size, int32_t num_pages,
                                       const int32_t *prefix_lens, const void *tree_k, const void *tree_v,
                                       const int32_t *parents, const int32_t *n_nodes, void *out,
                                       const jf_shape *shape, void *workspace, size_t workspace_bytes,
                                       int32_t *status, jf_stream_t stream) {
    if (page_size <= 0) return JF_ERR_SHAPE;
    return attention_call(q, k_pages, v_pages, block_table, page_size, num_pages, prefix_lens, tree_k, tree_v,
                          parents, n_nodes, out, shape, workspace, workspace_bytes, status, stream);
}

JF_API int32_t jf_tree_verify(const void *logits, const int32_t *tree_tokens, const int32_t *parents,
                              const int32_t *n_nodes, int32_t *accept_len_out, int32_t *accept_path_out,
                              int32_t *argmax_out, const jf_shape *shape, int32_t max_depth, void *workspace,
                              size_t workspace_bytes, int32_t *status, jf_stream_t stream) {
    if (!logits || !tree_tokens || !parents || !n_nodes || !accept_len_out || !accept_path_out || !shape ||
        !workspace)
        return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, true, false);
    if (sc != JF_OK) return sc;
    if (max_depth < 0) return JF_ERR_SHAPE;
    if (!aligned16(logits) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return JF_ERR_ALIGN;
    if (workspace_bytes < jf_workspace_bytes(shape)) return JF_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
    const int sms = num_sms_cached(dev);
    if (sms <= 0) return JF_ERR_CUDA;
    const Layout L = layout_of(shape, sms);          // the argmax chunking for this device
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    if (launch_argmax(L, reinterpret_cast<const __nv_bfloat16 *>(logits), n_nodes, ws, s) != cudaSuccess)
        return JF_ERR_CUDA;
    if (launch_accept_walk(L, tree_tokens, parents, n_nodes, accept_len_out, accept_path_out, argmax_out, max_depth,
                           ws, status, s) != cudaSuccess)
        return JF_ERR_CUDA;
    return JF_OK;
}

JF_API int32_t jf_tree_verify_sample(const void *target_logits, const void *draft_logits, const int32_t *tree_tokens,
                                     const int32_t *parents, const int32_t *n_nodes, float temperature,
                                     uint64_t seed, uint64_t offset, int32_t *accept_len_out,
                                     int32_t *accept_path_out, int32_t *next_token_out, const jf_shape *shape,
                                     int32_t max_depth, void *workspace, size_t workspace_bytes, int32_t *status,
                                     jf_stream_t stream) {
    if (!target_logits || !draft_logits || !tree_tokens || !parents || !n_nodes || !accept_len_out ||
        !accept_path_out || !next_token_out || !shape || !workspace)
        return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, true, false);
    if (sc != JF_OK) return sc;
    if (max_depth < 0 || !(temperature > 0.0f) || isinf(temperature)) return JF_ERR_SHAPE;
    if (!aligned16(target_logits) || !aligned16(draft_logits) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return JF_ERR_ALIGN;
    if (workspace_bytes < jf_workspace_bytes(shape)) return JF_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
    const int sms = num_sms_cached(dev);
    if (sms <= 0) return JF_ERR_CUDA;
    const Layout L = layout_of(shape, sms);
    SampleArgs a{};
    a.target = reinterpret_cast<const __nv_bfloat16 *>(target_logits);
    a.draft = reinterpret_cast<const __nv_bfloat16 *>(draft_logits);
    a.tokens = tree_tokens;
    a.parents = parents;
    a.n_nodes = n_nodes;
    a.accept_len = accept_len_out;
    a.accept_path = accept_path_out;
    a.next_token = next_token_out;
    a.status = status;
    a.k2 = 1.4426950408889634f / temperature;
    a.seed = seed;
    a.offset = offset;
    a.max_depth = max_depth;
    if (launch_sample(L, a, reinterpret_cast<uint8_t *>(workspace), sms, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return JF_ERR_CUDA;
    return JF_OK;
}

JF_API int32_t jf_tree_score(const void *draft_logits, const int32_t *tree_tokens, const int32_t *parents,
                             const int32_t *n_nodes, float temperature, int32_t top_k, int32_t budget,
                             float *node_logprob_out, float *path_logprob_out, int32_t *topk_token_out,
                             float *topk_logprob_out, int32_t *cand_parent_out, int32_t *cand_token_out,
                             float *cand_score_out, const jf_shape *shape, void *workspace, size_t workspace_bytes,
                             int32_t *status, jf_stream_t stream) {
    if (!draft_logits || !tree_tokens || !parents || !n_nodes || !node_logprob_out || !path_logprob_out || !shape ||
        !workspace)
        return JF_ERR_NULL;
    if (top_k > 0 && (!topk_token_out || !topk_logprob_out)) return JF_ERR_NULL;
    if (budget > 0 && (!cand_parent_out || !cand_token_out || !cand_score_out)) return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, true, false);
    if (sc != JF_OK) return sc;
    if (!(temperature > 0.0f) || isinf(temperature)) return JF_ERR_SHAPE;
    if (top_k < 0 || top_k > kScoreMaxK || budget < 0 || (budget > 0 && top_k == 0) ||
        (long long)budget > (long long)shape->max_nodes * top_k)
        return JF_ERR_SHAPE;
    if (!aligned16(draft_logits) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return JF_ERR_ALIGN;
    if (workspace_bytes < jf_workspace_bytes(shape)) return JF_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
    const int sms = num_sms_cached(dev);
    if (sms <= 0) return JF_ERR_CUDA;
    const Layout L = layout_of(shape, sms);
    ScoreArgs a{};
    a.draft = reinterpret_cast<const __nv_bfloat16 *>(draft_logits);
    a.tokens = tree_tokens;
    a.parents = parents;
    a.n_nodes = n_nodes;
    a.node_lp = node_logprob_out;
    a.path_lp = path_logprob_out;
    a.topk_token = topk_token_out;
    a.topk_lp = topk_logprob_out;
    a.cand_parent = cand_parent_out;
    a.cand_token = cand_token_out;
    a.cand_score = cand_score_out;
    a.status = status;
    a.k2 = 1.4426950408889634f / temperature;
    a.top_k = top_k;
    a.budget = budget;
    if (launch_score(L, a, reinterpret_cast<uint8_t *>(workspace), sms, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return JF_ERR_CUDA;
    return JF_OK;
}

JF_API int32_t jf_tree_commit_kv(const void *tree_k, const void *tree_v, const int32_t *n_nodes,
                                 const int32_t *accept_len, const int32_t *accept_path, void *k_cache,
                                 void *v_cache, int32_t *prefix_lens, const jf_shape *shape, int32_t max_depth,
                                 int32_t *status, jf_stream_t stream) {
    if (!tree_k || !tree_v || !n_nodes || !accept_len || !accept_path || !k_cache || !v_cache || !prefix_lens ||
        !shape)
        return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, false, true);
    if (sc != JF_OK) return sc;
    if (max_depth < 0) return JF_ERR_SHAPE;
    if (!aligned16(tree_k) || !aligned16(tree_v) || !aligned16(k_cache) || !aligned16(v_cache)) return JF_ERR_ALIGN;
    const Layout L = layout_of(shape);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_commit_kv(L, reinterpret_cast<const __nv_bfloat16 *>(tree_k),
                         reinterpret_cast<const __nv_bfloat16 *>(tree_v), n_nodes, accept_len, accept_path,
                         reinterpret_cast<__nv_bfloat16 *>(k_cache), reinterpret_cast<__nv_bfloat16 *>(v_cache),
                         prefix_lens, max_depth, status, s) != cudaSuccess)
        return JF_ERR_CUDA;
    return JF_OK;
}

JF_API int32_t jf_tree_commit_kv_paged(const void *tree_k, const void *tree_v, const int32_t *n_nodes,
                                       const int32_t *accept_len, const int32_t *accept_path, void *k_pages,
                                       void *v_pages, const int32_t *block_table, int32_t page_size,
                                       int32_t num_pages, int32_t *prefix_lens, const jf_shape *shape,
                                       int32_t max_depth, int32_t *status, jf_stream_t stream) {
    if (!tree_k || !tree_v || !n_nodes || !accept_len || !accept_path || !k_pages || !v_pages || !block_table ||
        !prefix_lens || !shape)
        return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, false, true);
    if (sc != JF_OK) return sc;
    if (max_depth < 0) return JF_ERR_SHAPE;
    int page_lg = 0;
    while (page_lg < 31 && (1 << page_lg) < page_size) ++page_lg;
    if (page_size < 8 || page_size > kBN || (1 << page_lg) != page_size || shape->prefix_cap % page_size ||
        num_pages < 1 || (long long)num_pages * page_size > 0x7FFFFFFFll)
        return JF_ERR_SHAPE;
    if (!aligned16(tree_k) || !aligned16(tree_v) || !aligned16(k_pages) || !aligned16(v_pages)) return JF_ERR_ALIGN;
    const Layout L = layout_of(shape);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_commit_kv(L, reinterpret_cast<const __nv_bfloat16 *>(tree_k),
                         reinterpret_cast<const __nv_bfloat16 *>(tree_v), n_nodes, accept_len, accept_path,
                         reinterpret_cast<__nv_bfloat16 *>(k_pages), reinterpret_cast<__nv_bfloat16 *>(v_pages),
                         prefix_lens, max_depth, status, s, block_table, page_lg, num_pages) != cudaSuccess)
        return JF_ERR_CUDA;
    return JF_OK;
}

// ------------------------------------------------ allocation-free verify
// Scratch for jf_tree_verify_noalloc: lives in the library's own device
// memory, so the call needs no caller workspace and allocates nothing.
static __device__ __align__(256) uint8_t g_noalloc_scratch[JF_NOALLOC_SCRATCH_BYTES];

// Current driver context (CUcontext), through the runtime's driver entry
// point query so that the library needs no link-time dependency on libcuda.
static void *current_context() {
    typedef CUresult (*CtxGetFn)(CUcontext *);
    static CtxGetFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetFn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device and context (a reset device gets a new context, and the module
// a new address). In host code the symbol's name is only a host-side
// stand-in, so the kernels must be given this address instead.
static uint8_t *noalloc_scratch(int dev) {
    static std::mutex mu;
    static uint8_t *addr[64] = {nullptr};
    static void *ctx[64] = {nullptr};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    void *cur = current_context();
    if (!addr[dev] || cur != ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = reinterpret_cast<uint8_t *>(p);
        ctx[dev] = current_context();   // the lookup may have created the primary context
    }
    return addr[dev];
}

JF_API int32_t jf_tree_verify_noalloc(const void *logits, const int32_t *tree_tokens, const int32_t *parents,
                                      const int32_t *n_nodes, int32_t *accept_len_out, int32_t *accept_path_out,
                                      int32_t *argmax_out, const jf_shape *shape, int32_t max_depth,
                                      int32_t *status, jf_stream_t stream) {
    if (!logits || !tree_tokens || !parents || !n_nodes || !accept_len_out || !accept_path_out || !shape)
        return JF_ERR_NULL;
    const int32_t sc = check_shape(shape, true, false);
    if (sc != JF_OK) return sc;
    if (max_depth < 0) return JF_ERR_SHAPE;
    if (!aligned16(logits)) return JF_ERR_ALIGN;
    // rows * chunks int2 must fit the array: refuse what cannot fit even at
    // one chunk per 76800 elements before any CUDA call, then check the
    // chunking of this device exactly
    const long long rows = (long long)shape->batch * shape->max_nodes;
    if (rows * ceil_div(shape->vocab, kArgmaxMaxChunk) * (long long)sizeof(int2) > (long long)JF_NOALLOC_SCRATCH_BYTES)
        return JF_ERR_SHAPE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JF_ERR_CUDA;
    const int sms = num_sms_cached(dev);
    if (sms <= 0) return JF_ERR_CUDA;
    Layout L = layout_of(shape, sms);
    const size_t need = sizeof(int2) * (size_t)L.B * L.Nmax * L.chunks;
    if (need > (size_t)JF_NOALLOC_SCRATCH_BYTES) return JF_ERR_SHAPE;
    uint8_t *scratch = noalloc_scratch(dev);
    if (!scratch) return JF_ERR_CUDA;
    L.amp_off = 0;   // the verify region starts at the array's first byte
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_argmax(L, reinterpret_cast<const __nv_bfloat16 *>(logits), n_nodes, scratch, s) != cudaSuccess)
        return JF_ERR_CUDA;
    if (launch_accept_walk(L, tree_tokens, parents, n_nodes, accept_len_out, accept_path_out, argmax_out, max_depth,
                           scratch, status, s) != cudaSuccess)
        return JF_ERR_CUDA;
    return JF_OK;
}

JF_API uint64_t jf_kernel_launch_count(void) { return g_launches.load(); }

JF_API int32_t jf_trace_kernels(jf_event_t *events, int32_t capacity) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace_events = (events && capacity > 0) ? events : nullptr;
    g_trace_capacity = g_trace_events ? capacity : 0;
    g_trace_count = 0;
    return JF_OK;
}

JF_API int32_t jf_trace_count(void) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    return g_trace_count;
}

JF_API const char *jf_trace_name(int32_t k) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (k < 0 || k >= g_trace_count || k >= 4096) return nullptr;
    return g_trace_names[k];
}

}  // extern "C"
