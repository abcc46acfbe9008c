// jf_prep.cu - the two small kernels around tree attention:
//
//  tree_prep_kernel     (before attention) one block per sequence validates
//                       the tree and builds per-node ancestor bitmasks; one
//                       more block plans the split-KV work items.
//  split_combine_kernel (after attention) merges the fp32 partials of query
//                       tiles that were split over several CTAs.
//
// Ancestor mask ("JetFlow: Scaling Speculative Decoding with Parallel Tree
// Drafting", blog, section "What JetFlow Does Differently": a node attends to
// its ancestors, never to siblings or descendants): bit j of mask[b][i] is
// set iff j is i or an ancestor of i. It is built by pointer jumping in
// shared memory: after round r each node holds its ancestors at distance
// < 2^r and a pointer to its 2^r-th ancestor, so 8 rounds cover any tree of
// up to 256 nodes.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kMaskWords = kMaxNodes / 32;   // 8
constexpr int kHistBins = 256;

__device__ __forceinline__ int tiles_of(const Layout &L, int P, int n, int qt, int Pcap) {
    const bool ok = n >= 1 && n <= L.Nmax && P >= 0 && P <= Pcap;
    const int node0 = qt * L.NB;
    if (!ok || node0 >= n) return 0;
    const int n_hi = min(node0 + L.NB, n);
    return ceil_div(P, kBN) + ceil_div(n_hi, kBN);
}

__device__ __forceinline__ int split_begin(int T, int ns, int s) { return (int)(((long long)s * T) / ns); }

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ int block_exclusive_scan(int v, int *out_excl, int *sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kPrepThreads / 32 ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kPrepThreads / 32) sh[lane] = w;
    }
    __syncthreads();
    const int total = sh[kPrepThreads / 32 - 1];
    *out_excl = x - v + (warp > 0 ? sh[warp - 1] : 0);
    __syncthreads();
    return total;
}

__device__ void build_sequence(const Layout &L, const AttnArgs &a, int b) {
    __shared__ uint32_t anc[2][kMaxNodes][kMaskWords];
    __shared__ int jmp[2][kMaxNodes];
    const int i = threadIdx.x;
    const int N = L.Nmax;
    const int n = a.n_nodes[b];
    const int P = a.prefix_lens[b];
    const int *par = a.parents + (size_t)b * N;
    bool bad = !(n >= 1 && n <= N && P >= 0 && P <= L.Pcap);
    int p = -1;
    if (!bad && i < n) {
        p = par[i];
        bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
    }
    bad = __syncthreads_or(bad);
    SeqInfo *seq = reinterpret_cast<SeqInfo *>(a.ws + L.seq_off);
    if (i == 0) seq[b] = SeqInfo{P, n, bad ? 1 : 0, 0};
    if (bad) {
        if (i == 0) set_status(a.status, JF_STATUS_BAD_TREE);
        // every output row of a malformed sequence becomes NaN
        const size_t per_seq = (size_t)N * L.Hq * L.D;
        uint32_t *o = reinterpret_cast<uint32_t *>(a.out + (size_t)b * per_seq);
        for (size_t k = i; k < per_seq / 2; k += blockDim.x) o[k] = 0x7FC07FC0u;
        return;
    }
    const int W = ceil_div(N, 32);
    if (i < kMaxNodes) {
        for (int w = 0; w < kMaskWords; ++w) anc[0][i][w] = 0u;
        if (i < n) anc[0][i][i >> 5] = 1u << (i & 31);
        jmp[0][i] = (i < n) ? p : -1;
    }
    __syncthreads();
    int cur = 0;
    for (int round = 0; round < 8; ++round) {
        const int nxt = cur ^ 1;
        int live = 0;
        if (i < kMaxNodes) {
            const int j = jmp[cur][i];
            for (int w = 0; w < W; ++w) anc[nxt][i][w] = anc[cur][i][w] | (j >= 0 ? anc[cur][j][w] : 0u);
            const int jj = j >= 0 ? jmp[cur][j] : -1;
            jmp[nxt][i] = jj;
            live = jj >= 0;
        }
        cur = nxt;
        if (!__syncthreads_or(live)) break;
    }
    if (i < N) {
        uint32_t *dst = reinterpret_cast<uint32_t *>(a.ws + L.mask_off) + ((size_t)b * N + i) * L.W4;
        for (int w = 0; w < L.W4; ++w) dst[w] = (w < W && i < n) ? anc[cur][i][w] : 0u;
    }
}

// Plan: per query tile T tiles (prefix tiles + tree tiles it needs); split
// size tps = max(kMinTilesPerSplit, ceil(total / num_ctas)); a tile of T
// tiles gets ceil(T / tps) near-equal splits. Items are ordered longest
// first (counting sort on length) for the atomic work queue, so short
// remainders fill in behind long items.
__device__ void plan(const Layout &L, const AttnArgs &a) {
    __shared__ int sh[32];
    __shared__ int hist[kHistBins];
    __shared__ int s_total;
    const int tid = threadIdx.x;
    const int nbq = L.B * L.QT;
    int local = 0;
    for (int k = tid; k < nbq; k += blockDim.x) {
        const int b = k / L.QT, qt = k % L.QT;
        local += tiles_of(L, a.prefix_lens[b], a.n_nodes[b], qt, L.Pcap);
    }
    int excl;
    const int total = L.Hkv * block_exclusive_scan(local, &excl, sh);
    const int tps = max(kMinTilesPerSplit, ceil_div(total, max(1, a.num_ctas)));
    for (int k = tid; k < kHistBins; k += blockDim.x) hist[k] = 0;
    __syncthreads();

    int2 *qtab = reinterpret_cast<int2 *>(a.ws + L.qtab_off);
    Item *items = reinterpret_cast<Item *>(a.ws + L.items_off);
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + L.plan_off);
    auto bin_of = [&](int size) { return min(size, kHistBins - 1); };

    // pass 1: split counts, histogram of item lengths, slot bases
    int slot_run = 0;
    for (int base = 0; base < L.n_qtiles; base += blockDim.x) {
        const int q = base + tid;
        int ns = 0, T = 0;
        if (q < L.n_qtiles) {
            const int b = q / (L.Hkv * L.QT);
            const int qt = q % L.QT;
            T = tiles_of(L, a.prefix_lens[b], a.n_nodes[b], qt, L.Pcap);
            ns = T > 0 ? ceil_div(T, tps) : 0;
            for (int s = 0; s < ns; ++s)
                atomicAdd(&hist[bin_of(split_begin(T, ns, s + 1) - split_begin(T, ns, s))], 1);
        }
        int ex;
        const int tot = block_exclusive_scan(ns > 1 ? ns : 0, &ex, sh);
        if (q < L.n_qtiles) qtab[q] = make_int2(ns, slot_run + ex);
        slot_run += tot;
    }
    __syncthreads();
    // descending-length starting offsets
    if (tid == 0) {
        int run = 0;
        for (int k = kHistBins - 1; k >= 0; --k) {
            const int c = hist[k];
            hist[k] = run;
            run += c;
        }
        s_total = run;
    }
    __syncthreads();
    // pass 2: scatter items
    for (int q = tid; q < L.n_qtiles; q += blockDim.x) {
        const int b = q / (L.Hkv * L.QT);
        const int qt = q % L.QT;
        const int T = tiles_of(L, a.prefix_lens[b], a.n_nodes[b], qt, L.Pcap);
        const int ns = T > 0 ? ceil_div(T, tps) : 0;
        for (int s = 0; s < ns; ++s) {
            const int b0 = split_begin(T, ns, s), b1 = split_begin(T, ns, s + 1);
            const int pos = atomicAdd(&hist[bin_of(b1 - b0)], 1);
            if (pos < L.max_items) items[pos] = Item{q, b0, b1, s};
        }
    }
    __syncthreads();
    if (tid == 0) {
        const int n_items = min(s_total, L.max_items);
        if (s_total > L.max_items) set_status(a.status, JF_STATUS_TIMEOUT);   // cannot happen: bound proven
        *hdr = PlanHeader{n_items, 0, tps, total};
    }
}

__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(const Layout L, const AttnArgs a) {
    if ((int)blockIdx.x < L.B)
        build_sequence(L, a, blockIdx.x);
    else
        plan(L, a);
}

// One block per query tile; a warp per stacked row. Partials of split s are
// (O_s unnormalised, m_s, l_s) with m in the exp2 domain:
//   O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
template <int D>
__global__ void __launch_bounds__(256) split_combine_kernel(const Layout L, const AttnArgs a) {
    const int q = blockIdx.x;
    const int2 qi = reinterpret_cast<const int2 *>(a.ws + L.qtab_off)[q];
    const int ns = qi.x, base = qi.y;
    if (ns <= 1) return;
    const int b = q / (L.Hkv * L.QT);
    const int rem = q % (L.Hkv * L.QT);
    const int kh = rem / L.QT, qt = rem % L.QT;
    const SeqInfo si = reinterpret_cast<const SeqInfo *>(a.ws + L.seq_off)[b];
    if (si.bad) return;
    const float2 *ml = reinterpret_cast<const float2 *>(a.ws + L.ml_off);
    const float *op = reinterpret_cast<const float *>(a.ws + L.opart_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int E = D / 32;   // elements per lane
    for (int r = warp; r < kBM; r += 8) {
        const int node = qt * L.NB + r / L.G;
        if (node >= si.n_nodes) break;              // rows are ordered by node
        const int head = kh * L.G + r % L.G;
        float M = -__int_as_float(0x7f800000);
        for (int s = lane; s < ns; s += 32) M = fmaxf(M, ml[(size_t)(base + s) * kBM + r].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if (M == -__int_as_float(0x7f800000)) M = 0.f;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float Lsum = 0.f;
        for (int s = 0; s < ns; ++s) {
            const size_t row = (size_t)(base + s) * kBM + r;
            const float2 mls = ml[row];
            const float w = ex2_approx(mls.x - M);
            Lsum += w * mls.y;
            const float *src = op + row * D + lane * E;
            if constexpr (E == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                acc[0] += w * v.x; acc[1] += w * v.y;
            }
        }
        const float inv = 1.0f / Lsum;
        __nv_bfloat16 *dst = a.out + (((size_t)b * L.Nmax + node) * L.Hq + head) * D + lane * E;
        if constexpr (E == 4) {
            uint2 w;
            w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2 *>(dst) = w;
        } else {
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
    }
}

}  // namespace

cudaError_t launch_tree_prep(const Layout &L, const AttnArgs &a, cudaStream_t s) {
    trace_begin("tree_prep", s);
    tree_prep_kernel<<<L.B + 1, kPrepThreads, 0, s>>>(L, a);
    cudaError_t e = cudaGetLastError();
    trace_end(s);
    return e;
}

cudaError_t launch_split_combine(const Layout &L, const AttnArgs &a, cudaStream_t s) {
    trace_begin("split_combine", s);
    if (L.D == 128)
        split_combine_kernel<128><<<L.n_qtiles, 256, 0, s>>>(L, a);
    else
        split_combine_kernel<64><<<L.n_qtiles, 256, 0, s>>>(L, a);
    cudaError_t e = cudaGetLastError();
    trace_end(s);
    return e;
}

}  // namespace jf
