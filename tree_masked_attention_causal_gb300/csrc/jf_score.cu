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
//                      cover 256 levels), writes the top-k, and selects the
//                      budget best (node, rank) candidates by path score: a
//                      radix select of the budget-th key, then a bitonic
//                      sort of the selected ones, in shared memory.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kScoreThreads = 256;           // = kMaxNodes: one thread per node in the tree kernel
constexpr int kScoreCands = kMaxNodes * kScoreMaxK;   // candidates of the expansion, at most
constexpr int kScoreMaxChunks = 4;           // chunks a row in the scan, at most

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

// The elements of one vector per lane (8 bf16, indices idx0 ..) that clear
// the bar (the list's last entry), inserted one at a time in (element,
// lane) order. Once the list is full few vectors get here; it is out of
// line, since the scan's loop runs faster with less code (measured: a
// copy inlined at every call site, or a list filled from the first
// vectors and a bar shared between warps, were slower).
__device__ __noinline__ WarpTop warp_take(WarpTop t, uint4 vec, bool live, int idx0) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        const uint32_t wj = (j >> 1) == 0 ? vec.x : (j >> 1) == 1 ? vec.y : (j >> 1) == 2 ? vec.z : vec.w;
        const float zj = __uint_as_float((j & 1) ? (wj & 0xFFFF0000u) : (wj << 16));
        const int ix = idx0 + j;
        unsigned cand = __ballot_sync(full, live && ahead(zj, ix, t.thr_v, t.thr_i));
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

// The kScoreMaxK best of two lists sorted by `ahead` into (lv, li): a
// bitonic half-cleaner on lv ++ reverse(cv), then a bitonic merge of the
// better half (static indices throughout, so the lists stay in registers).
__device__ __forceinline__ void merge_top(float (&lv)[kScoreMaxK], int (&li)[kScoreMaxK], const float (&cv)[kScoreMaxK],
                                          const int (&ci)[kScoreMaxK]) {
#pragma unroll
    for (int q = 0; q < kScoreMaxK; ++q) {
        const float bv = cv[kScoreMaxK - 1 - q];
        const int bi = ci[kScoreMaxK - 1 - q];
        if (ahead(bv, bi, lv[q], li[q])) {
            lv[q] = bv;
            li[q] = bi;
        }
    }
#pragma unroll
    for (int stride = kScoreMaxK / 2; stride > 0; stride >>= 1) {
#pragma unroll
        for (int q = 0; q < kScoreMaxK; ++q) {
            if ((q & stride) == 0 && ahead(lv[q + stride], li[q + stride], lv[q], li[q])) {
                const float tv = lv[q];
                const int ti = li[q];
                lv[q] = lv[q + stride];
                li[q] = li[q + stride];
                lv[q + stride] = tv;
                li[q + stride] = ti;
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
    const int lane = tid & 31;
    const unsigned full = 0xffffffffu;
    WarpTop wt{kNegInf, -1, kNegInf, -1};
    // the loop bound is the same for the whole block, so every lane reaches
    // every ballot; lanes past the chunk's end take part with live = false
    for (int k0b = 0; k0b < nvec; k0b += kArgmaxThreads * kArgmaxVecs) {
        const int k0 = k0b + tid;
        uint4 v[kArgmaxVecs];
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            if (k < nvec) v[u] = ld_stream(src + k);
        }
#pragma unroll
        for (int u = 0; u < kArgmaxVecs; ++u) {
            const int k = k0 + u * kArgmaxThreads;
            const bool live = k < nvec;                       // warp-uniform loop: every lane takes the ballots
            float vm = kNegInf;
            if (live) {
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
            }
            // a vector whose largest entry reaches the bar may hold entries for the list
            if (want_top && __any_sync(full, live && !(vm < wt.thr_v))) wt = warp_take(wt, v[u], live, e0 + 8 * k);
        }
    }
    __shared__ float2 sacc[kArgmaxThreads / 32];
    __shared__ float swv[kArgmaxThreads / 32];
    __shared__ int swi[kArgmaxThreads / 32];
    const int warp = tid >> 5;
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
    // the block's kScoreMaxK best: each round every warp offers the head of
    // its list, the best offer is written out, and its warp drops its head
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
            top_v[slot * kScoreMaxK + r] = bv;
            top_i[slot * kScoreMaxK + r] = bi;
        }
        if (warp == bw && bi >= 0) {                          // the winning warp drops its head
            const float nv = __shfl_down_sync(full, wt.ev, 1);
            const int ni = __shfl_down_sync(full, wt.ei, 1);
            wt.ev = lane < kScoreMaxK - 1 ? nv : kNegInf;
            wt.ei = lane < kScoreMaxK - 1 ? ni : -1;
        }
    }
}

struct ScoreShared {
    int par[kMaxNodes];
    float lp[kMaxNodes];         // node_lp, then path sums
    float lp2[kMaxNodes];
    int anc[kMaxNodes], anc2[kMaxNodes];
    float ms[kMaxNodes][2];      // row max, log2 sum
    // the expansion's candidates (node * K + rank): order key, score, token
    uint32_t cand_key[kScoreCands];
    float cand_s[kScoreCands];
    int cand_tok[kScoreCands];
    // the selected ones, to sort
    uint32_t sel_key[kScoreCands];
    int sel_c[kScoreCands];
    int hist[kScoreThreads], tie_base[kScoreThreads];
    int sel_digit, sel_rest, n_sel;
};

__global__ void __launch_bounds__(kScoreThreads)
    score_tree_kernel(const Layout L, const ScoreArgs a, const float2 *__restrict__ lse_part,
                      const float *__restrict__ top_v, const int *__restrict__ top_i, int chunks) {
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
        const float2 *pr = lse_part + (seq + i) * chunks;
        float2 acc = make_float2(kNegInf, 0.f);
        for (int ch = 0; ch < chunks; ++ch) acc = lse_merge(acc, pr[ch], a.k2);
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
    // this node's top-k: its chunks' lists (at most kScoreMaxChunks, each
    // loaded whole with 16-byte loads) merged in chunk (index) order
    float lv[kScoreMaxK];
    int li[kScoreMaxK];
#pragma unroll
    for (int s = 0; s < kScoreMaxK; ++s) {
        lv[s] = kNegInf;
        li[s] = -1;
    }
    if (K > 0 && i < n) {
        for (int ch = 0; ch < chunks; ++ch) {
            const size_t slot = ((seq + i) * chunks + ch) * kScoreMaxK;
            float cv[kScoreMaxK];
            int ci[kScoreMaxK];
#pragma unroll
            for (int q = 0; q < kScoreMaxK / 4; ++q) {
                const float4 v4 = *reinterpret_cast<const float4 *>(top_v + slot + 4 * q);
                const int4 i4 = *reinterpret_cast<const int4 *>(top_i + slot + 4 * q);
                cv[4 * q] = v4.x; cv[4 * q + 1] = v4.y; cv[4 * q + 2] = v4.z; cv[4 * q + 3] = v4.w;
                ci[4 * q] = i4.x; ci[4 * q + 1] = i4.y; ci[4 * q + 2] = i4.z; ci[4 * q + 3] = i4.w;
            }
            merge_top(lv, li, cv, ci);
        }
    }
    // outputs, and the expansion's candidates with an order-preserving key:
    // larger score -> larger key, no candidate -> 0
    const float m = i < n ? sh.ms[i][0] : 0.f, l2 = i < n ? sh.ms[i][1] : 0.f;
    const bool want = a.budget > 0 && K > 0;
#pragma unroll
    for (int s = 0; s < kScoreMaxK; ++s) {
        if (s < K && i < Nmax) {
            const bool ok = i < n && li[s] >= 0;
            const float v = ok ? ((lv[s] - m) * a.k2 - l2) * ln2 : kNaN;
            a.topk_token[(seq + i) * K + s] = ok ? li[s] : -1;
            a.topk_lp[(seq + i) * K + s] = v;
            if (want) {
                const float sc = path + v;
                const uint32_t u = __float_as_uint(sc);
                sh.cand_key[i * K + s] = (ok && sc == sc) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
                sh.cand_s[i * K + s] = sc;
                sh.cand_tok[i * K + s] = ok ? li[s] : -1;
            }
        }
    }
    if (!want) return;
    __syncthreads();
    // The budget-th largest key T by a radix select (four 8-bit digits,
    // shared-memory histograms); then every candidate above T, and those at
    // T in (node, rank) order until the budget is met, are compacted and
    // sorted (bitonic) best first: larger score, then lower (node, rank).
    const int total = Nmax * K;
    uint32_t prefix = 0, mask = 0;
    int want_rank = a.budget;                                  // 1-based rank of T among the candidates
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        sh.hist[i] = 0;                                        // 256 bins, one per thread
        __syncthreads();
        for (int c = i; c < total; c += kScoreThreads) {
            const uint32_t key = sh.cand_key[c];
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
            if (i < Nmax && sh.cand_key[i * K + s] == T) ++my_ties;
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
        const uint32_t key = sh.cand_key[i * K + s];
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
    int C = 1;
    while (C < nsel) C <<= 1;
    for (int k = nsel + i; k < C; k += kScoreThreads) {
        sh.sel_key[k] = 0u;
        sh.sel_c[k] = 0x7FFFFFFF;
    }
    __syncthreads();
    auto before = [](uint32_t ka, int ca, uint32_t kb, int cb) { return ka > kb || (ka == kb && ca < cb); };
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
            a.cand_token[o] = sh.cand_tok[c];
            a.cand_score[o] = sh.cand_s[c];
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
    // at most kScoreMaxChunks chunks a row, so that each node's merge loads
    // a few whole lists (the argmax cuts more when rows are few)
    int chunk = L.chunk, chunks = L.chunks;
    if (chunks > kScoreMaxChunks) {
        chunk = (int)align_up((size_t)ceil_div(L.V, kScoreMaxChunks), kArgmaxGranule);
        chunks = ceil_div(L.V, chunk);
    }
    float2 *lse_part = reinterpret_cast<float2 *>(ws + L.lse_off);
    float *top_v = reinterpret_cast<float *>(ws + L.topk_off);
    int *top_i = reinterpret_cast<int *>(ws + L.topk_off + sizeof(float) * kScoreMaxK * (size_t)rows * L.chunks);
    trace_begin("score_chunk", s);
    score_chunk_kernel<<<dim3(chunks, rows), kArgmaxThreads, 0, s>>>(a.draft, a.n_nodes, lse_part, top_v, top_i,
                                                                     L.Nmax, L.V, chunk, chunks, a.k2,
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
                           static_cast<const float *>(top_v), static_cast<const int *>(top_i), chunks);
    trace_end(s);
    return e;
}

}  // namespace jf
