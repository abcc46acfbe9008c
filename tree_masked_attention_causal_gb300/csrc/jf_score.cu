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
//                      argmax (at most 4 chunks a row), the chunks of one
//                      row forming one thread-block cluster. Each CTA
//                      reduces its chunk to (max z, sum 2^((z - max)
//                      log2(e) / T)) and, when asked, its kScoreMaxK
//                      largest entries (the lower index first on ties):
//                      while it reads, every entry at or above a running
//                      bound on the chunk's kScoreMaxK-th entry (taken from
//                      the threads' maxima) is kept in shared memory, and
//                      at the end the few kept entries are ranked. CTA 0
//                      of the cluster merges the chunks' normalisers and
//                      lists and writes the row's top_k log-probabilities.
//  score_tree_kernel   one block per sequence, one thread per node, a
//                      programmatic dependent of the scan. Before the scan
//                      completes it validates the tree and loads each
//                      node's token logit; after, it sums the path by
//                      pointer jumping (8 rounds cover 256 levels) and
//                      selects the budget best (node, rank) candidates by
//                      path score: a radix select of the budget-th key,
//                      then a bitonic sort of the selected ones, in shared
//                      memory.
#include "jf_cluster.cuh"

namespace jf {
namespace {

constexpr int kScoreThreads = 256;           // = kMaxNodes: one thread per node in the tree kernel
constexpr int kScoreCands = kMaxNodes * kScoreMaxK;   // candidates of the expansion, at most
constexpr int kScoreMaxChunks = 4;           // chunks a row in the scan, at most
constexpr int kScoreFastCap = 128;           // expansion candidates ranked directly, at most
constexpr int kScoreKeepCap = 256;           // a chunk's candidates ranked directly, at most
constexpr int kScoreTieCap = 256;            // candidates in the budget's bucket ranked directly, at most
static_assert(kScoreTieCap <= kScoreThreads, "one tie candidate per thread");

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

// A warp's kScoreMaxK best so far, sorted by `ahead`: lane l < kScoreMaxK
// holds entry l; thr is entry kScoreMaxK - 1, the bar a new element must
// clear.
struct WarpTop {
    float ev;
    int ei;
    float thr_v;
    int thr_i;
};

// The elements of one vector per lane (8 bf16, indices idx0 ..) that reach
// floor_v and clear the bar (the list's last entry), inserted one at a
// time in (element, lane) order. Out of line: few vectors get here.
__device__ __noinline__ WarpTop warp_take(WarpTop t, uint4 vec, bool live, int idx0, float floor_v) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        const uint32_t wj = (j >> 1) == 0 ? vec.x : (j >> 1) == 1 ? vec.y : (j >> 1) == 2 ? vec.z : vec.w;
        const float zj = __uint_as_float((j & 1) ? (wj & 0xFFFF0000u) : (wj << 16));
        const int ix = idx0 + j;
        unsigned cand = __ballot_sync(full, live && zj >= floor_v && ahead(zj, ix, t.thr_v, t.thr_i));
        while (cand) {
            const int src = __ffs(cand) - 1;
            cand &= cand - 1;
            const float x = __shfl_sync(full, zj, src);
            const int xi = __shfl_sync(full, ix, src);
            if (!ahead(x, xi, t.thr_v, t.thr_i)) continue;        // the bar has risen past it
            const bool stays_ahead = lane < kScoreMaxK && !ahead(x, xi, t.ev, t.ei);
            const int pos = __popc(__ballot_sync(full, stays_ahead));
            const float pv = __shfl_up_sync(full, t.ev, 1);
            const int pi = __shfl_up_sync(full, t.ei, 1);
            if (lane < kScoreMaxK && lane > pos) {
                t.ev = pv;
                t.ei = pi;
            }
            if (lane == pos) {
                t.ev = x;
                t.ei = xi;
            }
            t.thr_v = __shfl_sync(full, t.ev, kScoreMaxK - 1);
            t.thr_i = __shfl_sync(full, t.ei, kScoreMaxK - 1);
        }
    }
    return t;
}

// A bound T that the chunk's kScoreMaxK-th largest entry cannot be below:
// the two largest thread maxima of every warp are distinct entries of the
// chunk, kScoreMaxK of them over the block, so their minimum will do. Each
// warp's pair only grows as the scan goes on, so a bound taken from older
// values of some warps is still a bound.
static_assert(2 * (kArgmaxThreads / 32) == kScoreMaxK, "two thread maxima per warp make the bound");

// The largest of a vector's 8 bf16 entries (NaN only if all are NaN).
__device__ __forceinline__ float vm_of(uint4 v) {
    const float a = fmaxf(fmaxf(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u)),
                          fmaxf(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)));
    const float b = fmaxf(fmaxf(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u)),
                          fmaxf(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u)));
    return fmaxf(a, b);
}

// The second largest of the warp's values (the largest counted once).
__device__ __forceinline__ float warp_second(float x) {
    const unsigned full = 0xffffffffu;
    float m1 = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m1 = fmaxf(m1, __shfl_xor_sync(full, m1, o));
    const int first = __ffs(__ballot_sync(full, x == m1)) - 1;
    float m2 = (int)(threadIdx.x & 31) == first ? -__builtin_huge_valf() : x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m2 = fmaxf(m2, __shfl_xor_sync(full, m2, o));
    return m2;
}

// The scan's candidates: each thread keeps up to kThreadCands of its own
// in a strided slot of shared memory, counting in a register.
constexpr int kThreadCands = 8;
constexpr int kScoreCap = kArgmaxThreads * kThreadCands;
__shared__ float s_cand_v[kScoreCap];
__shared__ int s_cand_i[kScoreCap];

__device__ __forceinline__ float bound_of(const volatile float *sbound) {
    float T = sbound[0];
#pragma unroll
    for (int w = 1; w < kArgmaxThreads / 32; ++w) T = fminf(T, sbound[w]);
    return T;
}

// The chunk's kScoreMaxK best by a second pass over the vectors whose
// maximum reaches T: a sorted list per warp, then the block's best taken
// from the warps' lists one at a time and stored at dst_v / dst_i (a CTA's
// slot in its cluster's CTA 0). Called by the whole block; out of line, so
// that the scan keeps its registers.
__device__ __noinline__ void chunk_lists(const uint4 *src, int nvec, int e0, float T, float my_max, uint32_t dst_v,
                                         uint32_t dst_i) {
    constexpr float kNegInf = -__builtin_huge_valf();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    __shared__ float swv[kArgmaxThreads / 32];
    __shared__ int swi[kArgmaxThreads / 32];
    WarpTop wt{kNegInf, -1, kNegInf, -1};
    const bool mine = my_max >= T;
    if (__any_sync(full, mine)) {
        // the loop bound is the same for the whole warp, so every lane
        // reaches every ballot; other lanes take part with live = false
        for (int k0b = 0; k0b < nvec; k0b += kArgmaxThreads * kArgmaxVecs) {
            const int k0 = k0b + tid;
            uint4 v[kArgmaxVecs];
#pragma unroll
            for (int u = 0; u < kArgmaxVecs; ++u) {
                const int k = k0 + u * kArgmaxThreads;
                if (mine && k < nvec) v[u] = ld_stream(src + k);
            }
#pragma unroll
            for (int u = 0; u < kArgmaxVecs; ++u) {
                const int k = k0 + u * kArgmaxThreads;
                const bool live = mine && k < nvec;
                const float vm = live ? vm_of(v[u]) : kNegInf;
                if (__any_sync(full, live && vm >= T && !(vm < wt.thr_v)))
                    wt = warp_take(wt, v[u], live, e0 + 8 * k, T);
            }
        }
    }
    // the block's kScoreMaxK best: each round every warp offers the
    // head of its list, the best offer is stored, and its warp drops
    // its head
    for (int r = 0; r < kScoreMaxK; ++r) {
        if (lane == 0) {
            swv[warp] = wt.ev;
            swi[warp] = wt.ei;
        }
        __syncthreads();
        float bv = swv[0];
        int bi = swi[0], bw = 0;
        for (int w2 = 1; w2 < kArgmaxThreads / 32; ++w2)
            if (ahead(swv[w2], swi[w2], bv, bi)) {
                bv = swv[w2];
                bi = swi[w2];
                bw = w2;
            }
        __syncthreads();
        if (tid == 0) {
            st_cluster(dst_v + 4 * r, __float_as_uint(bv));
            st_cluster(dst_i + 4 * r, (uint32_t)bi);
        }
        if (warp == bw && bi >= 0) {                      // the winning warp drops its head
            const float nv = __shfl_down_sync(full, wt.ev, 1);
            const int ni = __shfl_down_sync(full, wt.ei, 1);
            wt.ev = lane < kScoreMaxK - 1 ? nv : kNegInf;
            wt.ei = lane < kScoreMaxK - 1 ? ni : -1;
        }
    }
}

__global__ void __launch_bounds__(kArgmaxThreads)
    score_chunk_kernel(const __nv_bfloat16 *__restrict__ draft, const int32_t *__restrict__ n_nodes,
                       float2 *__restrict__ row_lse, int32_t *__restrict__ topk_token, float *__restrict__ topk_lp,
                       int K, int Nmax, int V, int chunk, float k2) {
    pdl_launch_dependents();
    const int row = blockIdx.y;
    const int b = row / Nmax, node = row - b * Nmax;
    const int n = n_nodes[b];
    if (n < 1 || n > Nmax || node >= n) return;              // padding row (the whole cluster)
    const int tid = threadIdx.x;
    const int e0 = blockIdx.x * chunk;
    const int nvec = (min(V, e0 + chunk) - e0) >> 3;
    const uint4 *src = reinterpret_cast<const uint4 *>(draft + (size_t)row * V + e0);
    constexpr float kNegInf = -__builtin_huge_valf();
    const bool want_top = K > 0;
    const int lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    __shared__ float2 sacc[kArgmaxThreads / 32];
    __shared__ float sbound[kArgmaxThreads / 32];
    __shared__ int s_over;
    volatile float *vbound = sbound;
    float2 acc = make_float2(kNegInf, 0.f);
    // Candidates: the entries at or above the bound known when their vector
    // is reduced, appended to shared memory. Every entry of the chunk's top
    // kScoreMaxK is one, whatever the order the warps run in.
    float T = kNegInf;
    int ncand = 0;
    for (int k0b = 0; k0b < nvec; k0b += kArgmaxThreads * kArgmaxVecs) {
        const int k0 = k0b + tid;
        uint4 v[kArgmaxVecs];
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            if (k < nvec) v[u] = ld_stream(src + k);
        }
        if (want_top && k0b > 0) {                            // raise this warp's part of the bound
            const float m2 = warp_second(acc.x);                // (with the loads in flight)
            if (lane == 0) vbound[warp] = m2;
            T = bound_of(vbound);
        }
        if (want_top && k0b == 0) {                           // the first bound, from the first vectors
            float tm = kNegInf;
#pragma unroll
            for (int u = 0; u < kArgmaxVecs; ++u)
                if (k0 + u * kArgmaxThreads < nvec) tm = fmaxf(tm, vm_of(v[u]));
            const float m2 = warp_second(tm);
            if (lane == 0) vbound[warp] = m2;
            if (tid == 0) s_over = 0;
            __syncthreads();
            T = bound_of(vbound);
        }
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            float vm = kNegInf;
            if (k < nvec) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                float z[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    z[2 * j] = __uint_as_float(w[j] << 16);
                    z[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                }
                vm = z[0];
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
                if (want_top && vm >= T) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (z[j] >= T) {
                            if (ncand < kThreadCands) {
                                s_cand_v[ncand * kArgmaxThreads + tid] = z[j];
                                s_cand_i[ncand * kArgmaxThreads + tid] = e0 + 8 * k + j;
                            }
                            ++ncand;
                        }
                    }
                }
            }
        }
    }
    const float my_max = acc.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float2 other = make_float2(__shfl_xor_sync(full, acc.x, o), __shfl_xor_sync(full, acc.y, o));
        acc = lse_merge(acc, other, k2);
    }
    if (want_top && nvec > 0) {                               // this warp's final pair
        const float m2 = warp_second(my_max);
        if (lane == 0) vbound[warp] = m2;
    }
    if (want_top && ncand > kThreadCands) s_over = 1;
    if (lane == 0) sacc[warp] = acc;
    __syncthreads();
    // The row's chunks are one cluster: each CTA stores its (max, sum) and
    // its kScoreMaxK best into CTA 0's shared memory, which then writes the
    // row's normaliser and its top_k.
    __shared__ float2 s_lse_all[kScoreMaxChunks];
    __shared__ float s_all_v[kScoreMaxChunks * kScoreMaxK];
    __shared__ int s_all_i[kScoreMaxChunks * kScoreMaxK];
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    if (tid == 0) {
        float2 t = sacc[0];
        for (int w2 = 1; w2 < kArgmaxThreads / 32; ++w2) t = lse_merge(t, sacc[w2], k2);
        const uint32_t dst = map_to_rank(smem_u32(&s_lse_all[crank]), 0);
        st_cluster(dst, __float_as_uint(t.x));
        st_cluster(dst + 4, __float_as_uint(t.y));
    }
    T = want_top && nvec > 0 ? bound_of(vbound) : kNegInf;    // every warp's final pair
    // only the candidates at or above the final bound can rank below
    // kScoreMaxK: those are compacted, then (when few) each is ranked among
    // them
    __shared__ int s_keep;
    __shared__ float s_kv[kScoreCap];
    __shared__ int s_ki[kScoreCap];
    const bool slots = want_top && (nvec == 0 || s_over == 0);
    if (slots) {
        if (tid == 0) s_keep = 0;
        __syncthreads();
        for (int q = 0; q < ncand; ++q) {                     // this thread's own
            const float x = s_cand_v[q * kArgmaxThreads + tid];
            if (x >= T) {
                const int at = atomicAdd(&s_keep, 1);
                s_kv[at] = x;
                s_ki[at] = s_cand_i[q * kArgmaxThreads + tid];
            }
        }
        __syncthreads();
    }
    const int keep = slots ? s_keep : kScoreCap + 1;
    const uint32_t dst_v = map_to_rank(smem_u32(&s_all_v[crank * kScoreMaxK]), 0);
    const uint32_t dst_i = map_to_rank(smem_u32(&s_all_i[crank * kScoreMaxK]), 0);
    if (!want_top) {
    } else if (keep <= kScoreKeepCap) {
        for (int t = tid; t < keep; t += kArgmaxThreads) {
            const float x = s_kv[t];
            const int xi = s_ki[t];
            int rank = 0;
#pragma unroll 4
            for (int q = 0; q < keep; ++q) rank += ahead(s_kv[q], s_ki[q], x, xi) ? 1 : 0;
            if (rank < kScoreMaxK) {
                st_cluster(dst_v + 4 * rank, __float_as_uint(x));
                st_cluster(dst_i + 4 * rank, (uint32_t)xi);
            }
        }
        if (tid >= keep && tid < kScoreMaxK) {                // fewer entries than the list holds
            st_cluster(dst_v + 4 * tid, __float_as_uint(kNegInf));
            st_cluster(dst_i + 4 * tid, (uint32_t)-1);
        }
    } else {
        // More candidates than the slots keep (many entries equal at the
        // top of the chunk), or more than are worth ranking one by one (a
        // chunk too short for the bound): the lists pass.
        chunk_lists(src, nvec, e0, T, my_max, dst_v, dst_i);
    }
    cluster_sync_all();
    if (crank != 0) return;
    // CTA 0: the row's normaliser (chunks merged in order) as (max, log2 sum)
    float2 rl = s_lse_all[0];
    for (uint32_t c = 1; c < csize; ++c) rl = lse_merge(rl, s_lse_all[c], k2);
    const float l2 = log2f(rl.y);
    if (tid == 0) row_lse[row] = make_float2(rl.x, l2);
    if (!want_top) return;
    // the row's top_k: each real entry of the chunks' lists ranked among them
    const int total = (int)csize * kScoreMaxK;
    const bool real = tid < total && s_all_i[tid] >= 0;
    const int nreal = __syncthreads_count(real);
    const float ln2 = 0.69314718055994531f;
    if (real) {
        const float x = s_all_v[tid];
        const int xi = s_all_i[tid];
        int rank = 0;
        for (int q = 0; q < total; ++q) rank += (s_all_i[q] >= 0 && ahead(s_all_v[q], s_all_i[q], x, xi)) ? 1 : 0;
        if (rank < K) {
            topk_token[(size_t)row * K + rank] = xi;
            topk_lp[(size_t)row * K + rank] = ((x - rl.x) * k2 - l2) * ln2;
        }
    }
    if (tid >= nreal && tid < K) {                            // fewer entries than asked for
        topk_token[(size_t)row * K + tid] = -1;
        topk_lp[(size_t)row * K + tid] = __builtin_nanf("");
    }
}

struct ScoreShared {
    int par[kMaxNodes];
    float lp[kMaxNodes];         // node_lp, then path sums
    float lp2[kMaxNodes];
    int anc[kMaxNodes], anc2[kMaxNodes];
    float ms[kMaxNodes][2];      // row max, log2 sum
    // the expansion's candidates (node * K + rank): order key, score, token
    // stored rank-major: candidate (node u, rank s) at s * kScoreThreads + u,
    // so that a thread's entries fall in distinct banks
    uint32_t cand_key[kScoreCands];
    float cand_s[kScoreCands];
    int cand_tok[kScoreCands];
    // the selected ones, to sort
    uint32_t sel_key[kScoreCands];
    int sel_c[kScoreCands];
    int hist[kScoreThreads], tie_base[kScoreThreads];
    int sel_digit, sel_rest, n_sel, n_tie;
    uint32_t red_min[kScoreThreads / 32], red_max[kScoreThreads / 32];
    int red_cnt[kScoreThreads / 32];
};

__global__ void __launch_bounds__(kScoreThreads, 1)
    score_tree_kernel(const Layout L, const ScoreArgs a, const float2 *__restrict__ row_lse) {
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
    // Everything the scan wrote for this node, requested at once: its row's
    // normaliser (max, log2 sum) and, for the expansion, its K entries (the
    // scan wrote every one: NaN and -1 where a row has fewer).
    const bool want = a.budget > 0 && K > 0;
    int tok[kScoreMaxK];
    float v[kScoreMaxK];
    {
        const bool node = want && i < n;
        const int32_t *tp = a.topk_token + (seq + i) * K;
        const float *vp = a.topk_lp + (seq + i) * K;
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            const bool ok = node && s < K;
            tok[s] = ok ? __ldcg(tp + s) : -1;
            v[s] = ok ? __ldcg(vp + s) : kNaN;
        }
    }
    if (i < n) {
        const float2 rl = __ldcg(row_lse + seq + i);
        sh.ms[i][0] = rl.x;
        sh.ms[i][1] = rl.y;
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
        int up = -1;
        if (i < n) {
            const int j = ca[i];
            nxt[i] = j >= 0 ? cur[i] + cur[j] : cur[i];
            up = j >= 0 ? ca[j] : -1;
            na[i] = up;
        }
        const bool more = __syncthreads_or(up >= 0);
        float *t = cur;
        cur = nxt;
        nxt = t;
        int *ta = ca;
        ca = na;
        na = ta;
        if (!more) break;                                      // every path is summed
    }
    const float path = i < n ? cur[i] : kNaN;
    if (i < Nmax) {
        a.path_lp[seq + i] = path;
        if (i >= n) a.node_lp[seq + i] = kNaN;
    }
    // this node's top-k, written by the scan (padding rows get none), and
    // the expansion's candidates with an order-preserving key: larger score
    // -> larger key, no candidate -> 0
    if (i < Nmax && i >= n) {
        for (int s = 0; s < K; ++s) {
            a.topk_token[(seq + i) * K + s] = -1;
            a.topk_lp[(seq + i) * K + s] = kNaN;
        }
    }
    uint32_t ck[kScoreMaxK];                                   // this thread's keys, also in registers
#pragma unroll
    for (int s = 0; s < kScoreMaxK; ++s) ck[s] = 0u;
    if (want && i < Nmax) {
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            if (s < K) {
                const float sc = path + v[s];
                const uint32_t u = __float_as_uint(sc);
                ck[s] = (tok[s] >= 0 && sc == sc) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
                sh.cand_key[s * kScoreThreads + i] = ck[s];
                sh.cand_s[s * kScoreThreads + i] = sc;
                sh.cand_tok[s * kScoreThreads + i] = tok[s];
            }
        }
    }
    if (!want) return;
    __syncthreads();
    auto before = [](uint32_t ka, int ca, uint32_t kb, int cb) { return ka > kb || (ka == kb && ca < cb); };
    // Appends (key, c) where pred holds, one shared-memory atomic per warp:
    // at the front of sel_* (count n_sel) or from its back (count n_tie).
    const int lane = i & 31;
    auto append = [&](bool pred, bool back, uint32_t key, int c) {
        const unsigned m = __ballot_sync(0xffffffffu, pred);
        if (m == 0u) return;
        const int first = __ffs(m) - 1;
        int base = 0;
        if (lane == first) base = atomicAdd(back ? &sh.n_tie : &sh.n_sel, __popc(m));
        base = __shfl_sync(0xffffffffu, base, first);
        if (pred) {
            int at = base + __popc(m & ((1u << lane) - 1u));
            if (back) at = kScoreCands - 1 - at;
            sh.sel_key[at] = key;
            sh.sel_c[at] = c;
        }
    };
    // Each selected candidate's place in the output is its rank among the
    // selected: the number ahead of it (larger key, then lower (node,
    // rank)). With few real candidates, every one is selected and ranked.
    auto place = [&](int nsel) {
        // `per` threads (neighbouring lanes) count the ranks of one candidate
        // over interleaved parts of the list; the same number of rounds for
        // every lane, so that the lanes of a group reduce together.
        const int per = nsel <= kScoreThreads / 4 ? 4 : nsel <= kScoreThreads / 2 ? 2 : 1;
        const int groups = kScoreThreads / per, part = i % per;
        for (int e0 = 0; e0 < nsel; e0 += groups) {
            const int e = e0 + i / per;
            uint32_t key = 0u;
            int c = 0, rank = 0;
            if (e < nsel) {
                key = sh.sel_key[e];
                c = sh.sel_c[e];
#pragma unroll 4
                for (int f = part; f < nsel; f += per) rank += before(sh.sel_key[f], sh.sel_c[f], key, c) ? 1 : 0;
            }
            for (int o = 1; o < per; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
            if (e < nsel && part == 0 && rank < a.budget) {
                const size_t o = (size_t)b * a.budget + rank;
                a.cand_parent[o] = c / K;
                const int at = (c % K) * kScoreThreads + c / K;
                a.cand_token[o] = sh.cand_tok[at];
                a.cand_score[o] = sh.cand_s[at];
            }
        }
        for (int r = nsel + i; r < a.budget; r += kScoreThreads) {   // fewer candidates than the budget
            const size_t o = (size_t)b * a.budget + r;
            a.cand_parent[o] = -1;
            a.cand_token[o] = -1;
            a.cand_score[o] = kNaN;
        }
    };
    // Thread i's candidates marked in selm to the front of sel_*, those in
    // tiem to its back, in (node, rank) order: each thread's two counts
    // packed in one int, one block-wide exclusive scan gives the offsets.
    auto compact = [&](uint32_t selm, uint32_t tiem) {
        const int cnt = __popc(selm) | (__popc(tiem) << 16);   // each below 2^16
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) sh.red_cnt[i >> 5] = incl;
        __syncthreads();
        int off = incl - cnt, tot = 0;
        for (int w = 0; w < kScoreThreads / 32; ++w) {
            const int t = sh.red_cnt[w];
            off += w < (i >> 5) ? t : 0;
            tot += t;
        }
        int os = off & 0xFFFF, ot = off >> 16;
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            if ((selm >> s) & 1u) {
                sh.sel_key[os] = ck[s];
                sh.sel_c[os++] = i * K + s;
            }
            if ((tiem >> s) & 1u) {
                sh.sel_key[kScoreCands - 1 - ot] = ck[s];
                sh.sel_c[kScoreCands - 1 - ot++] = i * K + s;
            }
        }
        if (i == 0) {
            sh.n_sel = tot & 0xFFFF;
            sh.n_tie = tot >> 16;
        }
        __syncthreads();
    };
    uint32_t real = 0u;                                        // this thread's real candidates
#pragma unroll
    for (int s = 0; s < kScoreMaxK; ++s) real |= (s < K && ck[s] != 0u) ? 1u << s : 0u;
    if (__syncthreads_count(real != 0u) * K <= kScoreFastCap) {      // at most kScoreFastCap real ones
        compact(real, 0u);
        place(sh.n_sel);
        return;
    }
    if (a.budget <= kScoreFastCap) {
        // One pass of 256 equal buckets over the keys' range: every
        // candidate in a bucket above the budget-th key's bucket D is
        // selected, and those in D are ranked among themselves for the rest
        // (the selected then placed by rank). A crowded D (many equal keys)
        // takes the radix selection below.
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            if ((real >> s) & 1u) {
                kmin = min(kmin, ck[s]);
                kmax = max(kmax, ck[s]);
            }
        }
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        if (lane == 0) {
            sh.red_min[i >> 5] = kmin;
            sh.red_max[i >> 5] = kmax;
        }
        sh.hist[i] = 0;                                        // 256 bins, one per thread
        __syncthreads();
        for (int w = 0; w < kScoreThreads / 32; ++w) {
            kmin = min(kmin, sh.red_min[w]);
            kmax = max(kmax, sh.red_max[w]);
        }
        const uint32_t range = kmax - kmin;                    // some candidate is real here
        const int shift = max(0, 24 - __clz(range));           // (range >> shift) < 256
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s)
            if ((real >> s) & 1u) atomicAdd(&sh.hist[(ck[s] - kmin) >> shift], 1);
        __syncthreads();
        if (i < 32) {                                          // warp 0: the bucket holding rank budget
            int cnt[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {                      // lane l takes bins 255 - 8l .. 248 - 8l
                cnt[q] = sh.hist[255 - 8 * i - q];
                sum += cnt[q];
            }
            int incl = sum;                                    // lanes before: higher buckets
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (i >= o) incl += y;
            }
            int before_me = incl - sum, found = -1, rest = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (found < 0 && a.budget > before_me && a.budget <= before_me + cnt[q]) {
                    found = 255 - 8 * i - q;
                    rest = a.budget - before_me;
                }
                before_me += cnt[q];
            }
            const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
            if (hit) {
                const int src = __ffs(hit) - 1;
                found = __shfl_sync(0xffffffffu, found, src);
                rest = __shfl_sync(0xffffffffu, rest, src);
            }
            if (i == 0) {
                sh.sel_digit = found;                          // -1: fewer candidates than the budget
                sh.sel_rest = rest;
                sh.n_sel = 0;
                sh.n_tie = 0;
            }
        }
        __syncthreads();
        const int D = sh.sel_digit, need = sh.sel_rest;
        // selected ones to the front of sel_*, bucket D's to the back
        uint32_t selm = 0u, tiem = 0u;
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            const int bk = (int)((ck[s] - kmin) >> shift);
            if (((real >> s) & 1u) && (D < 0 || bk > D)) selm |= 1u << s;
            if (((real >> s) & 1u) && D >= 0 && bk == D) tiem |= 1u << s;
        }
        compact(selm, tiem);
        const int ntie = sh.n_tie;
        if (D < 0 || ntie <= kScoreTieCap) {                  // kScoreTieCap <= kScoreThreads: one each
            uint32_t key = 0u;
            int c = 0, rank = need;
            if (D >= 0 && i < ntie) {
                key = sh.sel_key[kScoreCands - 1 - i];
                c = sh.sel_c[kScoreCands - 1 - i];
                rank = 0;
                for (int f = 0; f < ntie; ++f)
                    rank += before(sh.sel_key[kScoreCands - 1 - f], sh.sel_c[kScoreCands - 1 - f], key, c) ? 1 : 0;
            }
            __syncthreads();                                   // the tie entries are read before any append
            append(rank < need, false, key, c);
            __syncthreads();
            place(sh.n_sel);
            return;
        }
        __syncthreads();
    }
    // The budget-th largest key T by a radix select (four 8-bit digits,
    // shared-memory histograms); then every candidate above T, and those at
    // T in (node, rank) order until the budget is met, are compacted and
    // sorted (bitonic) best first: larger score, then lower (node, rank).
    uint32_t prefix = 0, mask = 0;
    int want_rank = a.budget;                                  // 1-based rank of T among the candidates
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        sh.hist[i] = 0;                                        // 256 bins, one per thread
        __syncthreads();
#pragma unroll
        for (int s = 0; s < kScoreMaxK; ++s) {
            const uint32_t key = ck[s];
            if (key != 0u && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (i < 32) {                                          // warp 0: the digit holding rank want_rank
            int cnt[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {                      // lane l takes bins 255 - 8l .. 248 - 8l
                cnt[q] = sh.hist[255 - 8 * i - q];
                sum += cnt[q];
            }
            int incl = sum;                                    // lanes before: larger digits
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (i >= o) incl += y;
            }
            int before = incl - sum;
            int found = -1, rest = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (found < 0 && want_rank > before && want_rank <= before + cnt[q]) {
                    found = 255 - 8 * i - q;
                    rest = want_rank - before;
                }
                before += cnt[q];
            }
            const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
            if (hit) {
                const int src = __ffs(hit) - 1;
                found = __shfl_sync(0xffffffffu, found, src);
                rest = __shfl_sync(0xffffffffu, rest, src);
            }
            if (i == 0) {
                sh.sel_digit = found;
                sh.sel_rest = rest;
            }
        }
        __syncthreads();
        if (sh.sel_digit < 0) break;                           // fewer candidates than the budget
        prefix |= (uint32_t)sh.sel_digit << shift;
        mask |= 255u << shift;
        want_rank = sh.sel_rest;
        __syncthreads();
    }
    const bool short_list = sh.sel_digit < 0;                  // every real candidate is selected
    const uint32_t T = prefix;
    // ties at T: the first want_rank of them in (node, rank) order
    int my_ties = 0;
    if (!short_list)
        for (int s = 0; s < K; ++s)
            if (i < Nmax && sh.cand_key[s * kScoreThreads + i] == T) ++my_ties;
    // exclusive prefix of ties over threads (node order)
    sh.hist[i] = my_ties;
    __syncthreads();
    if (i < 32) {
        int part = 0;
        for (int q = 0; q < 8; ++q) part += sh.hist[8 * i + q];
        int incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (i >= o) incl += y;
        }
        int run = incl - part;
        for (int q = 0; q < 8; ++q) {
            const int c = sh.hist[8 * i + q];
            sh.tie_base[8 * i + q] = run;
            run += c;
        }
    }
    if (i == 0) sh.n_sel = 0;
    __syncthreads();
    int tie_rank = sh.tie_base[i];
    for (int s = 0; s < K && i < Nmax; ++s) {
        const uint32_t key = sh.cand_key[s * kScoreThreads + i];
        bool take = key != 0u && (short_list || key > T);
        if (!short_list && key == T) take = tie_rank++ < want_rank;
        if (take) {
            const int at = atomicAdd(&sh.n_sel, 1);
            sh.sel_key[at] = key;
            sh.sel_c[at] = i * K + s;
        }
    }
    __syncthreads();
    const int nsel = sh.n_sel;
    if (nsel <= kScoreFastCap) {
        place(nsel);
        return;
    }
    int C = 1;
    while (C < nsel) C <<= 1;
    for (int k = nsel + i; k < C; k += kScoreThreads) {
        sh.sel_key[k] = 0u;
        sh.sel_c[k] = 0x7FFFFFFF;
    }
    __syncthreads();
    for (int size = 2; size <= C; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = i; t < C / 2; t += kScoreThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const uint32_t kl = sh.sel_key[lo], kh = sh.sel_key[hi];
                const int cl = sh.sel_c[lo], ch2 = sh.sel_c[hi];
                if (up ? before(kh, ch2, kl, cl) : before(kl, cl, kh, ch2)) {
                    sh.sel_key[lo] = kh;
                    sh.sel_key[hi] = kl;
                    sh.sel_c[lo] = ch2;
                    sh.sel_c[hi] = cl;
                }
            }
            __syncthreads();
        }
    }
    for (int r = i; r < a.budget; r += kScoreThreads) {
        const size_t o = (size_t)b * a.budget + r;
        if (r < nsel) {
            const int c = sh.sel_c[r];
            a.cand_parent[o] = c / K;
            const int at = (c % K) * kScoreThreads + c / K;
            a.cand_token[o] = sh.cand_tok[at];
            a.cand_score[o] = sh.cand_s[at];
        } else {
            a.cand_parent[o] = -1;
            a.cand_token[o] = -1;
            a.cand_score[o] = kNaN;
        }
    }
}

}  // namespace

cudaError_t launch_score(const Layout &L, const ScoreArgs &a, uint8_t *ws, int sms, cudaStream_t s) {
    const int rows = L.B * L.Nmax;
    // at most kScoreMaxChunks chunks a row, one cluster (the argmax cuts
    // more when rows are few); one a row when the rows alone fill a wave,
    // so that each row's closing work (ranking, the cluster merge) is done
    // once
    int chunk = L.chunk, chunks = L.chunks;
    if (chunks > kScoreMaxChunks) {
        chunk = (int)align_up((size_t)ceil_div(L.V, kScoreMaxChunks), kArgmaxGranule);
        chunks = ceil_div(L.V, chunk);
    }
    if (L.V > 0 && rows >= kArgmaxCtasPerSm * sms) {
        chunk = (int)align_up((size_t)L.V, kArgmaxGranule);
        chunks = 1;
    }
    float2 *row_lse = reinterpret_cast<float2 *>(ws + L.lse_off);
    trace_begin("score_chunk", s);
    cudaLaunchConfig_t cc{};
    cc.gridDim = dim3(chunks, rows, 1);
    cc.blockDim = dim3(kArgmaxThreads, 1, 1);
    cc.stream = s;
    cudaLaunchAttribute ca[1];
    ca[0].id = cudaLaunchAttributeClusterDimension;
    ca[0].val.clusterDim.x = chunks;
    ca[0].val.clusterDim.y = 1;
    ca[0].val.clusterDim.z = 1;
    cc.attrs = ca;
    cc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cc, score_chunk_kernel, a.draft, a.n_nodes, row_lse, a.topk_token, a.topk_lp,
                                       a.top_k, L.Nmax, L.V, chunk, a.k2);
    trace_end(s);
    if (e != cudaSuccess) return e;
    // the tree kernel's shared-memory opt-in, once per device
    static bool smem_set[64] = {false};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!smem_set[dev]) {
        e = cudaFuncSetAttribute(score_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(ScoreShared));
        if (e != cudaSuccess) return e;
        smem_set[dev] = true;
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
    e = cudaLaunchKernelEx(&cfg, score_tree_kernel, L, a, static_cast<const float2 *>(row_lse));
    trace_end(s);
    return e;
}

}  // namespace jf
