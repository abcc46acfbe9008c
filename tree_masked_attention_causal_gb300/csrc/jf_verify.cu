// jf_verify.cu - greedy tree verification on sm_103a.
//
// The paper's section 2.1 "Background": the target verifies the drafted
// tokens in parallel and accepts the longest prefix that agrees with its own
// predictions. In a tree, node c is accepted iff its parent p is accepted and
// tokens[c] == argmax(logits[p]); the result is the deepest accepted node.
//
//  argmax_chunk_kernel  HBM-bound scan of the logits. Each CTA owns a chunk
//                       of one row: about 76800 bf16 (two chunks per row of
//                       151936, one wave of CTAs for 256 rows at 4 CTAs per
//                       SM), or shorter chunks when there are few rows, so
//                       that the grid still fills the SMs. Every thread
//                       streams 128-bit loads, 8 in flight, and keeps a
//                       running maximum over its vectors: a packed bf16x2
//                       NaN-propagating max per vector, plus the first
//                       vector that reached it (its index and its 8
//                       values, kept in registers). At the end it finds the
//                       exact first position in that vector. A block
//                       reduction on (value, index) writes the chunk's
//                       result.
//  accept_walk_kernel   one block per sequence, one thread per node. While
//                       the scan runs (programmatic launch) it validates the
//                       tree and builds every node's ancestor set by pointer
//                       jumping. After the scan: merges the chunk results
//                       (ties -> lowest index, the first NaN wins), checks
//                       each edge against the parent's argmax, accepts a
//                       node iff all edges on its root path agree (bit
//                       masks), and reduces (depth, -index) to the deepest
//                       accepted node, whose ancestor set gives the path.
#include "jf_common.cuh"

namespace jf {
namespace {

__device__ __forceinline__ bool is_nan_f(float x) { return x != x; }

// Max that propagates NaN (a NaN beats every number).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    return is_nan_f(a) ? a : (is_nan_f(b) ? b : fmaxf(a, b));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t hmax2_nan(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
    __nv_bfloat162 z = __hmax2_nan(x, y);
    return *reinterpret_cast<uint32_t *>(&z);
}

// Largest of the 8 bf16 of a vector, as fp32 (exact), NaN if any is NaN.
__device__ __forceinline__ float vec_max(const uint4 &v) {
    const uint32_t m2 = hmax2_nan(hmax2_nan(v.x, v.y), hmax2_nan(v.z, v.w));
    return fmax_nan(bf16_lo(m2), bf16_hi(m2));
}

// (a, ia) ranks before (b, ib): a NaN first, then the larger value, then
// the lower index (+0 == -0 compare equal).
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
    const bool an = is_nan_f(a), bn = is_nan_f(b);
    if (an != bn) return an;
    if (!an && a != b) return a > b;
    return ia < ib;
}

__global__ void __launch_bounds__(kArgmaxThreads, kArgmaxCtasPerSm)
    argmax_chunk_kernel(const __nv_bfloat16 *__restrict__ logits, const int32_t *__restrict__ n_nodes,
                        int2 *__restrict__ part, int Nmax, int V, int chunk, int chunks) {
    // A programmatic dependent of whatever the stream ran before: nothing is
    // read before that grid has completed, so only the launch overlaps it.
    pdl_wait_prior_grid();
    const int row = blockIdx.y;
    const int b = row / Nmax, i = row - b * Nmax;
    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * chunk;
    const int nvec = (min(V, e0 + chunk) - e0) >> 3;         // V % 8 == 0
    const uint4 *src = reinterpret_cast<const uint4 *>(logits + (size_t)row * V + e0);
    // The first vectors go out before the row is known to be real: a
    // padding row's logits exist too, and the latency of n_nodes overlaps
    // theirs.
    uint4 v[kArgmaxVecs];
#pragma unroll
    for (int u = 0; u < kArgmaxVecs; ++u) {
        const int k = tid + u * kArgmaxThreads;
        if (k < nvec) v[u] = ld_stream(src + k);
    }
    const int n = n_nodes[b];
    if (n < 1 || n > Nmax || i >= n) {                       // padding row
        pdl_launch_dependents();
        return;
    }
    float best = -__int_as_float(0x7f800000);
    int best_k = -1;
    uint4 best_v = make_uint4(0u, 0u, 0u, 0u);              // the vector that holds it
    for (int k0 = tid; k0 < nvec; k0 += kArgmaxThreads * kArgmaxVecs) {
        if (k0 != tid) {
#pragma unroll
            for (int u = 0; u < kArgmaxVecs; ++u) {
                const int k = k0 + u * kArgmaxThreads;
                if (k < nvec) v[u] = ld_stream(src + k);
            }
        }
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            if (k < nvec) {
                const float m = vec_max(v[u]);
                // strict: the first vector that reaches the maximum is kept;
                // a NaN replaces any number and is never replaced
                if (best_k < 0 || m > best || (is_nan_f(m) && !is_nan_f(best))) {
                    best = m;
                    best_k = k;
                    best_v = v[u];
                }
            }
        }
    }
    pdl_launch_dependents();
    // first element of the winning vector that equals the maximum
    int idx = 0x7FFFFFFF;
    if (best_k >= 0) {
        const uint32_t w4[4] = {best_v.x, best_v.y, best_v.z, best_v.w};
        const bool want_nan = is_nan_f(best);
#pragma unroll
        for (int q = 7; q >= 0; --q) {
            const float x = (q & 1) ? bf16_hi(w4[q >> 1]) : bf16_lo(w4[q >> 1]);
            if (want_nan ? is_nan_f(x) : (x == best)) idx = e0 + 8 * best_k + q;
        }
    }
    // block reduction on (value, index)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ranks_before(ob, oi, best, idx)) {
            best = ob;
            idx = oi;
        }
    }
    __shared__ float sv[kArgmaxThreads / 32];
    __shared__ int si[kArgmaxThreads / 32];
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        sv[warp] = best;
        si[warp] = idx;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kArgmaxThreads / 32; ++w)
            if (ranks_before(sv[w], si[w], best, idx)) {
                best = sv[w];
                idx = si[w];
            }
        part[(size_t)row * chunks + blockIdx.x] = make_int2(__float_as_int(best), idx);
    }
}

// (value, index) as one integer that orders like ranks_before: a NaN above
// every number, then the larger value (+0 == -0), then the lower index.
__device__ __forceinline__ unsigned long long rank_key(int2 x) {
    uint32_t u = static_cast<uint32_t>(x.x);
    uint32_t ord;
    if (is_nan_f(__int_as_float(x.x))) {
        ord = 0xFFFFFFFFu;
    } else {
        if (u == 0x80000000u) u = 0u;                      // -0 -> +0
        ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(x.y));
}

__global__ void __launch_bounds__(kMaxNodes)
    accept_walk_kernel(const int2 *__restrict__ part, const int32_t *__restrict__ tokens,
                       const int32_t *__restrict__ parents, const int32_t *__restrict__ n_nodes,
                       int32_t *__restrict__ accept_len, int32_t *__restrict__ accept_path,
                       int32_t *__restrict__ argmax_out, int Nmax, int chunks, int max_depth,
                       int32_t *status) {
    constexpr int W = kMaxNodes / 32;                       // words of a node mask
    __shared__ uint32_t anc[kMaxNodes][W];                  // node i and its ancestors
    __shared__ int jump[kMaxNodes];
    __shared__ int am[kMaxNodes];
    __shared__ unsigned long long best_key[kMaxNodes];      // merged chunk results
    __shared__ uint32_t ok_bits[W];                         // nodes whose edge to the parent agrees
    __shared__ int red[W];
    pdl_launch_dependents();        // whatever follows may start its prologue
    const int b = blockIdx.x, i = threadIdx.x;
    // Everything that depends on the tree alone is done before waiting for
    // the scan: validation, and every node's ancestor set and depth.
    const int n = n_nodes[b];
    const bool n_ok = n >= 1 && n <= Nmax;
    const bool real = n_ok && i < n;
    int p = -1, tok = 0;
    if (real) {
        p = parents[(size_t)b * Nmax + i];
        tok = tokens[(size_t)b * Nmax + i];
    }
    bool bad = !n_ok;
    if (real) bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
    best_key[i] = 0ull;
    bad = __syncthreads_or(bad);
    uint32_t m[W];
    int depth = 0;
    if (!bad) {
        // Pointer jumping: after round k, m holds the nodes on the path from
        // i up to (not including) its 2^k-th ancestor jump[i]; 8 rounds
        // cover any depth below 256.
#pragma unroll
        for (int w = 0; w < W; ++w) m[w] = (real && (i >> 5) == w) ? (1u << (i & 31)) : 0u;
        int up = real ? p : -1;
#pragma unroll
        for (int w = 0; w < W; ++w) anc[i][w] = m[w];
        jump[i] = up;
        __syncthreads();
#pragma unroll 1
        for (int round = 0; round < 8; ++round) {
            int up2 = -1;
            if (up >= 0) {
#pragma unroll
                for (int w = 0; w < W; ++w) m[w] |= anc[up][w];
                up2 = jump[up];
            }
            const bool more = __syncthreads_or(up2 >= 0);
#pragma unroll
            for (int w = 0; w < W; ++w) anc[i][w] = m[w];
            jump[i] = up2;
            up = up2;
            __syncthreads();
            if (!more) break;
        }
#pragma unroll
        for (int w = 0; w < W; ++w) depth += __popc(m[w]);
        depth -= 1;                                        // the node itself
    }
    pdl_wait_prior_grid();
    // Merge the chunk results. Up to 4 chunks per row: each node's thread
    // loads its entries together and keeps the best. More: the block's
    // threads share the sequence's n * chunks entries (node-major), four
    // loads in flight each, and keep the best per node with a shared-memory
    // atomic max on rank_key.
    unsigned long long mine = 0ull;
    if (chunks <= 4) {
        if (real) {
            const int2 *pr = part + ((size_t)b * Nmax + i) * chunks;
            int2 x[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (c < chunks) x[c] = __ldcg(pr + c);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const unsigned long long k = c < chunks ? rank_key(x[c]) : 0ull;
                mine = k > mine ? k : mine;
            }
        }
    } else {
        const int total = n_ok ? n * chunks : 0;
        const int2 *pb = part + (size_t)b * Nmax * chunks;
        for (int e0 = i; e0 < total; e0 += 4 * kMaxNodes) {
            int2 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (e0 + u * kMaxNodes < total) x[u] = __ldcg(pb + e0 + u * kMaxNodes);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * kMaxNodes;
                if (e < total) atomicMax(&best_key[e / chunks], rank_key(x[u]));
            }
        }
        __syncthreads();
        mine = best_key[i];
    }
    const int a = real ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(mine)) : -1;
    if (argmax_out && i < Nmax) argmax_out[(size_t)b * Nmax + i] = a;
    int32_t *path = accept_path + (size_t)b * (max_depth + 1);
    if (bad) {
        for (int k = i; k <= max_depth; k += blockDim.x) path[k] = -1;
        if (i == 0) {
            accept_len[b] = 0;
            set_status(status, JF_STATUS_BAD_TREE);
        }
        return;
    }
    am[i] = a;
    __syncthreads();
    // edge (p, i) agrees with the target; the root always does
    const bool edge = real && (i == 0 || tok == am[p]);
    const unsigned e = __ballot_sync(0xffffffffu, edge);
    if ((i & 31) == 0) ok_bits[i >> 5] = e;
    __syncthreads();
    // accepted iff every node on the root path (itself included) agrees
    bool acc = real;
#pragma unroll
    for (int w = 0; w < W; ++w) acc = acc && (m[w] & ~ok_bits[w]) == 0u;
    int key = acc ? (depth << 16) | (0xFFFF - i) : -1;      // deepest, then lowest index
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    if ((i & 31) == 0) red[i >> 5] = key;
    __syncthreads();
    int k = red[0];
#pragma unroll
    for (int w = 1; w < W; ++w) k = max(k, red[w]);
    const int best = 0xFFFF - (k & 0xFFFF);                 // the root is always accepted
    const int len = min(k >> 16, max_depth) + 1;
    // the path: the nodes of best's root path at depth < len, in depth order
    if (real && ((anc[best][i >> 5] >> (i & 31)) & 1u) && depth < len) path[depth] = i;
    for (int t = len + i; t <= max_depth; t += blockDim.x) path[t] = -1;
    if (i == 0) accept_len[b] = len;
}

}  // namespace

cudaError_t launch_argmax(const Layout &L, const __nv_bfloat16 *logits, const int32_t *n_nodes, uint8_t *ws,
                          cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.chunks, L.B * L.Nmax);
    cfg.blockDim = dim3(kArgmaxThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin("argmax_chunk", s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, argmax_chunk_kernel, logits, n_nodes,
                                       reinterpret_cast<int2 *>(ws + L.amp_off), (int)L.Nmax, (int)L.V,
                                       (int)L.chunk, (int)L.chunks);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(s);
    return e;
}

cudaError_t launch_accept_walk(const Layout &L, const int32_t *tokens, const int32_t *parents,
                               const int32_t *n_nodes, int32_t *accept_len, int32_t *accept_path,
                               int32_t *argmax_out, int32_t max_depth, uint8_t *ws, int32_t *status,
                               cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.B);
    cfg.blockDim = dim3(kMaxNodes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin("accept_walk", s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, accept_walk_kernel, reinterpret_cast<const int2 *>(ws + L.amp_off),
                                       tokens, parents, n_nodes, accept_len, accept_path, argmax_out, L.Nmax,
                                       L.chunks, max_depth, status);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(s);
    return e;
}

}  // namespace jf
