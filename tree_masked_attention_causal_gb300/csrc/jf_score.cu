// jf_score.cu - draft-side path scoring on sm_103a.
//
// "JetFlow: Scaling Speculative Decoding with Parallel Tree Drafting",
// section "What JetFlow Does Differently": a path's draft probability is
// the product of conditional distributions, each on the concrete ancestor
// tokens of its branch. Node u's row of draft logits holds the draft's
// distribution for u's children, q_u = softmax(z_u / T), so
//   node_lp[c] = log q_{parent(c)}(token_c),  path_lp[c] = sum over c's root
//   path of node_lp,
// and expanding the tree takes each node's most probable tokens, scored by
// path_lp[u] + log q_u(v), the best `budget` of them over the whole tree.
//
//  score_chunk_kernel  HBM-bound scan of the draft logits, chunked like the
//                      argmax: each CTA reduces its chunk of one row to
//                      (max z, sum 2^((z - max) log2(e) / T)) and, when
//                      asked, its kScoreMaxK largest entries (the lower
//                      index first on ties): a sorted list per thread,
//                      merged across the block one winner at a time.
//  score_tree_kernel   one block per sequence, one thread per node, a
//                      programmatic dependent of the scan. Before the scan
//                      completes it validates the tree and loads each
//                      node's token logit; after, it merges its row's
//                      chunks, sums the path by pointer jumping (8 rounds
//                      cover 256 levels), writes the top-k, and sorts every
//                      (node, rank) candidate by path score (bitonic, in
//                      shared memory) for the budgeted expansion.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kScoreThreads = 256;           // = kMaxNodes: one thread per node in the tree kernel
constexpr int kScoreCands = kMaxNodes * kScoreMaxK;   // candidates of the expansion, at most

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float2 lse_merge(float2 a, float2 b, float k2) {
    const float M = fmaxf(a.x, b.x);
    if (M == -__int_as_float(0x7f800000)) return make_float2(M, 0.f);
    return make_float2(M, a.y * ex2_approx((a.x - M) * k2) + b.y * ex2_approx((b.x - M) * k2));
}

// (a, ia) ranks before (b, ib): the larger value, then the lower index.
__device__ __forceinline__ bool ahead(float a, int ia, float b, int ib) {
    return a > b || (a == b && (unsigned)ia < (unsigned)ib);
}

// Insert (x, i) into a list sorted by `ahead`, if it ranks before its
// last entry. Entries arrive in increasing index, so strict > keeps the
// lower index ahead among equal values.
__device__ __forceinline__ void list_insert(float (&lv)[kScoreMaxK], int (&li)[kScoreMaxK], float x, int i) {
    if (!(x > lv[kScoreMaxK - 1])) return;
    bool placed = false;
#pragma unroll
    for (int s = kScoreMaxK - 1; s >= 0; --s) {
        if (!placed) {
            if (s > 0 && x > lv[s - 1]) {
                lv[s] = lv[s - 1];
                li[s] = li[s - 1];
            } else {
                lv[s] = x;
                li[s] = i;
                placed = true;
            }
        }
    }
}

__global__ void __launch_bounds__(kArgmaxThreads)
    score_chunk_kernel(const __nv_bfloat16 *__restrict__ draft, const int32_t *__restrict__ n_nodes,
                       float2 *__restrict__ lse_part, float *__restrict__ top_v, int *__restrict__ top_i, int Nmax,
                       int V, int chunk, int chunks, float k2, int want_top) {
    pdl_launch_dependents();
    const int row = blockIdx.y;
    const int b = row / Nmax, node = row - b * Nmax;
    const int n = n_nodes[b];
    if (n < 1 || n > Nmax || node >= n) return;              // padding row
    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * chunk;
    const int nvec = (min(V, e0 + chunk) - e0) >> 3;
    const uint4 *src = reinterpret_cast<const uint4 *>(draft + (size_t)row * V + e0);
    constexpr float kNegInf = -__builtin_huge_valf();
    float2 acc = make_float2(kNegInf, 0.f);
    float lv[kScoreMaxK];
    int li[kScoreMaxK];
#pragma unroll
    for (int s = 0; s < kScoreMaxK; ++s) {
        lv[s] = kNegInf;
        li[s] = -1;
    }
    for (int k0 = tid; k0 < nvec; k0 += kArgmaxThreads * kArgmaxVecs) {
        uint4 v[kArgmaxVecs];
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            if (k < nvec) v[u] = ld_stream(src + k);
        }
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            if (k < nvec) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                float z[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    z[2 * j] = __uint_as_float(w[j] << 16);
                    z[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                }
                float vm = z[0];
#pragma unroll
                for (int j = 1; j < 8; ++j) vm = fmaxf(vm, z[j]);
                if (vm > acc.x) {
                    acc.y *= ex2_approx((acc.x - vm) * k2);
                    acc.x = vm;
                }
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) s += ex2_approx((z[j] - acc.x) * k2);
                acc.y += s;
                if (want_top && vm > lv[kScoreMaxK - 1]) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) list_insert(lv, li, z[j], e0 + 8 * k + j);
                }
            }
        }
    }
    __shared__ float2 sacc[kArgmaxThreads / 32];
    __shared__ float swv[kArgmaxThreads / 32];
    __shared__ int swi[kArgmaxThreads / 32];
    const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, acc.x, o), __shfl_xor_sync(0xffffffffu, acc.y, o));
        acc = lse_merge(acc, other, k2);
    }
    if (lane == 0) sacc[warp] = acc;
    __syncthreads();
    const size_t slot = (size_t)row * chunks + blockIdx.x;
    if (tid == 0) {
        float2 t = sacc[0];
        for (int w2 = 1; w2 < kArgmaxThreads / 32; ++w2) t = lse_merge(t, sacc[w2], k2);
        lse_part[slot] = t;
    }
    if (!want_top) return;
    // the block's kScoreMaxK best: each round every thread offers the head
    // of its list, the best offer is written out, and its owner moves on
    for (int r = 0; r < kScoreMaxK; ++r) {
        float bv = lv[0];
        int bi = li[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ahead(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            swv[warp] = bv;
            swi[warp] = bi;
        }
        __syncthreads();
        bv = swv[0];
        bi = swi[0];
        for (int w2 = 1; w2 < kArgmaxThreads / 32; ++w2)
            if (ahead(swv[w2], swi[w2], bv, bi)) {
                bv = swv[w2];
                bi = swi[w2];
            }
        __syncthreads();
        if (tid == 0) {
            top_v[slot * kScoreMaxK + r] = bv;
            top_i[slot * kScoreMaxK + r] = bi;
        }
        if (bi >= 0 && li[0] == bi) {                         // the winner's owner drops its head
#pragma unroll
            for (int s = 0; s < kScoreMaxK - 1; ++s) {
                lv[s] = lv[s + 1];
                li[s] = li[s + 1];
            }
            lv[kScoreMaxK - 1] = kNegInf;
            li[kScoreMaxK - 1] = -1;
        }
    }
}

struct ScoreShared {
    int par[kMaxNodes];
    float lp[kMaxNodes];         // node_lp, then path sums
    float lp2[kMaxNodes];
    int anc[kMaxNodes], anc2[kMaxNodes];
    float ms[kMaxNodes][2];      // row max, log2 sum
    float cand_s[kScoreCands];   // the expansion's candidates: score
    int cand_k[kScoreCands];     //   and node * kScoreMaxK + rank (-1: none)
};

__global__ void __launch_bounds__(kScoreThreads)
    score_tree_kernel(const Layout L, const ScoreArgs a, const float2 *__restrict__ lse_part,
                      const float *__restrict__ top_v, const int *__restrict__ top_i) {
    extern __shared__ __align__(16) unsigned char s_raw[];
    ScoreShared &sh = *reinterpret_cast<ScoreShared *>(s_raw);
    const int b = blockIdx.x, i = threadIdx.x;
    const int Nmax = L.Nmax, V = L.V, K = a.top_k;
    const size_t seq = (size_t)b * Nmax;
    constexpr float kNaN = __builtin_nanf("");
    constexpr float kNegInf = -__builtin_huge_valf();
    const float ln2 = 0.69314718055994531f;
    // before the scan completes: the tree, and each node's token logit in its parent's row
    const int n = a.n_nodes[b];
    bool bad = n < 1 || n > Nmax;
    int p = -1;
    float ztok = kNegInf;
    if (!bad && i < n) {
        p = a.parents[seq + i];
        bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
        if (!bad && i > 0) {
            const int x = a.tokens[seq + i];
            if (x >= 0 && x < V)
                ztok = __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(a.draft) +
                                                       (seq + p) * (size_t)V + x) << 16);
        }
    }
    bad = __syncthreads_or(bad);
    pdl_wait_prior_grid();
    if (bad) {
        for (int k = i; k < Nmax; k += kScoreThreads) {
            a.node_lp[seq + k] = kNaN;
            a.path_lp[seq + k] = kNaN;
        }
        for (int k = i; k < Nmax * K; k += kScoreThreads) {
            a.topk_token[seq * K + k] = -1;
            a.topk_lp[seq * K + k] = kNaN;
        }
        for (int k = i; k < a.budget; k += kScoreThreads) {
            a.cand_parent[(size_t)b * a.budget + k] = -1;
            a.cand_token[(size_t)b * a.budget + k] = -1;
            a.cand_score[(size_t)b * a.budget + k] = kNaN;
        }
        if (i == 0) set_status(a.status, JF_STATUS_BAD_TREE);
        return;
    }
    // this node's row: its normaliser, merged from the chunks in order
    if (i < n) {
        const float2 *pr = lse_part + (seq + i) * L.chunks;
        float2 acc = make_float2(kNegInf, 0.f);
        for (int ch = 0; ch < L.chunks; ++ch) acc = lse_merge(acc, pr[ch], a.k2);
        sh.ms[i][0] = acc.x;
        sh.ms[i][1] = log2f(acc.y);
        sh.par[i] = p;
    }
    __syncthreads();
    // node_lp, then the path sums by pointer jumping: after round r a node
    // holds the sum over its 2^r nearest path nodes and points past them
    float lp = 0.f;
    if (i < n && i > 0) lp = ztok == kNegInf ? kNegInf : ((ztok - sh.ms[p][0]) * a.k2 - sh.ms[p][1]) * ln2;
    if (i < n) {
        a.node_lp[seq + i] = lp;
        sh.lp[i] = lp;
        sh.anc[i] = p;
    }
    __syncthreads();
    float *cur = sh.lp, *nxt = sh.lp2;
    int *ca = sh.anc, *na = sh.anc2;
    for (int r = 0; r < 8; ++r) {
        if (i < n) {
            const int j = ca[i];
            nxt[i] = j >= 0 ? cur[i] + cur[j] : cur[i];
            na[i] = j >= 0 ? ca[j] : -1;
        }
        __syncthreads();
        float *t = cur;
        cur = nxt;
        nxt = t;
        int *ta = ca;
        ca = na;
        na = ta;
    }
    const float path = i < n ? cur[i] : kNaN;
    if (i < Nmax) {
        a.path_lp[seq + i] = path;
        if (i >= n) a.node_lp[seq + i] = kNaN;
    }
    // this node's top-k: its chunks' lists merged in chunk (index) order
    if (K > 0 && i < Nmax) {
        float lv[kScoreMaxK];
        int li[kScoreMaxK];
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            lv[s] = kNegInf;
            li[s] = -1;
        }
        if (i < n) {
            for (int ch = 0; ch < L.chunks; ++ch) {
                const size_t slot = ((seq + i) * L.chunks + ch) * kScoreMaxK;
                for (int r = 0; r < kScoreMaxK; ++r) {
                    const int vi = top_i[slot + r];
                    if (vi < 0) break;
                    const float vv = top_v[slot + r];
                    if (!(vv > lv[kScoreMaxK - 1])) break;       // the list is sorted: nothing later enters
                    list_insert(lv, li, vv, vi);
                }
            }
        }
        const float m = i < n ? sh.ms[i][0] : 0.f, l2 = i < n ? sh.ms[i][1] : 0.f;
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            if (s < K) {
                const bool ok = i < n && li[s] >= 0;
                const float v = ok ? ((lv[s] - m) * a.k2 - l2) * ln2 : kNaN;
                a.topk_token[(seq + i) * K + s] = ok ? li[s] : -1;
                a.topk_lp[(seq + i) * K + s] = v;
                if (a.budget > 0) {
                    sh.cand_s[i * K + s] = ok ? path + v : kNegInf;
                    sh.cand_k[i * K + s] = ok ? i * kScoreMaxK + s : -1;
                }
            }
        }
    }
    if (a.budget <= 0 || K <= 0) return;
    // the expansion: bitonic sort of the Nmax * K candidates (padded to a
    // power of two), best first: larger score, then lower (node, rank)
    int C = 1;
    while (C < Nmax * K) C <<= 1;
    for (int k = Nmax * K + i; k < C; k += kScoreThreads) {
        sh.cand_s[k] = kNegInf;
        sh.cand_k[k] = -1;
    }
    __syncthreads();
    auto before = [](float sa, int ka, float sb, int kb) {  // a sorts ahead of b
        if (ka < 0 || kb < 0) return ka >= 0 && kb < 0;
        return sa > sb || (sa == sb && ka < kb);
    };
    for (int size = 2; size <= C; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = i; t < C / 2; t += kScoreThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const float sl = sh.cand_s[lo], shi = sh.cand_s[hi];
                const int kl = sh.cand_k[lo], kh = sh.cand_k[hi];
                const bool swap = up ? before(shi, kh, sl, kl) : before(sl, kl, shi, kh);
                if (swap) {
                    sh.cand_s[lo] = shi;
                    sh.cand_s[hi] = sl;
                    sh.cand_k[lo] = kh;
                    sh.cand_k[hi] = kl;
                }
            }
            __syncthreads();
        }
    }
    for (int r = i; r < a.budget; r += kScoreThreads) {
        const int key = r < C ? sh.cand_k[r] : -1;
        const size_t o = (size_t)b * a.budget + r;
        if (key >= 0) {
            const int u = key / kScoreMaxK, s = key - u * kScoreMaxK;
            a.cand_parent[o] = u;
            a.cand_token[o] = a.topk_token[(seq + u) * K + s];
            a.cand_score[o] = sh.cand_s[r];
        } else {
            a.cand_parent[o] = -1;
            a.cand_token[o] = -1;
            a.cand_score[o] = kNaN;
        }
    }
}

}  // namespace

cudaError_t launch_score(const Layout &L, const ScoreArgs &a, uint8_t *ws, cudaStream_t s) {
    const int rows = L.B * L.Nmax;
    float2 *lse_part = reinterpret_cast<float2 *>(ws + L.lse_off);
    float *top_v = reinterpret_cast<float *>(ws + L.topk_off);
    int *top_i = reinterpret_cast<int *>(ws + L.topk_off + sizeof(float) * kScoreMaxK * (size_t)rows * L.chunks);
    trace_begin("score_chunk", s);
    score_chunk_kernel<<<dim3(L.chunks, rows), kArgmaxThreads, 0, s>>>(a.draft, a.n_nodes, lse_part, top_v, top_i,
                                                                       L.Nmax, L.V, L.chunk, L.chunks, a.k2,
                                                                       a.top_k > 0 ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    trace_end(s);
    if (e != cudaSuccess) return e;
    static bool smem_set = false;
    if (!smem_set) {
        e = cudaFuncSetAttribute(score_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(ScoreShared));
        if (e != cudaSuccess) return e;
        smem_set = true;
    }
    trace_begin("score_tree", s);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(L.B, 1, 1);
    cfg.blockDim = dim3(kScoreThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(ScoreShared);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, score_tree_kernel, L, a, static_cast<const float2 *>(lse_part),
                           static_cast<const float *>(top_v), static_cast<const int *>(top_i));
    trace_end(s);
    return e;
}

}  // namespace jf
