// jf_prep.cu - the kernel that runs before tree attention.
//
//  tree_prep_kernel  one block per sequence validates the tree and builds
//                    per-node ancestor bitmasks; one more block plans the
//                    split-KV work items of the attention kernel.
//
// Ancestor mask ("JetFlow: Scaling Speculative Decoding with Parallel Tree
// Drafting", blog, section "What JetFlow Does Differently": a node attends to
// its ancestors, never to siblings or descendants): bit j of mask[b][i] is
// set iff j is i or an ancestor of i. It is built by pointer jumping in
// shared memory: after round r each node holds its ancestors at distance
// < 2^r and a pointer to its 2^r-th ancestor, so 8 rounds cover any tree of
// up to 256 nodes.
//
// The attention kernel is launched as a programmatic dependent of this one:
// its prologue overlaps this kernel, and it waits (griddepcontrol.wait)
// before it reads anything written here.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kMaskWords = kMaxNodes / 32;   // 8
constexpr int kHistBins = 256;

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ int block_exclusive_scan(int v, int *out_excl, int *sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kPrepThreads / 32 ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
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
    bool bad = !(n >= 1 && n <= N && P >= 0 && P <= L.Pcap);
    int p = -1;
    if (!bad && i < n) {
        p = a.parents[(size_t)b * N + i];
        bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
    }
    bad = __syncthreads_or(bad);
    SeqInfo *seq = reinterpret_cast<SeqInfo *>(a.ws + L.seq_off);
    if (i == 0) seq[b] = SeqInfo{P, n, bad ? 1 : 0, 0};
    if (bad) {
        if (i == 0) set_status(a.status, JF_STATUS_BAD_TREE);
        // every output row of a malformed sequence becomes NaN
        const size_t per_seq = (size_t)N * L.Hq * L.D;
        uint4 *o = reinterpret_cast<uint4 *>(a.out + (size_t)b * per_seq);
        const uint4 nan8 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
        for (size_t k = i; k < per_seq / 8; k += blockDim.x) o[k] = nan8;
        return;
    }
    const int W = ceil_div(N, 32);
    for (int w = 0; w < kMaskWords; ++w) anc[0][i][w] = 0u;
    if (i < n) anc[0][i][i >> 5] = 1u << (i & 31);
    jmp[0][i] = (i < n) ? p : -1;
    __syncthreads();
    int cur = 0;
    for (int round = 0; round < 8; ++round) {
        const int nxt = cur ^ 1;
        const int j = jmp[cur][i];
        for (int w = 0; w < W; ++w) anc[nxt][i][w] = anc[cur][i][w] | (j >= 0 ? anc[cur][j][w] : 0u);
        const int jj = j >= 0 ? jmp[cur][j] : -1;
        jmp[nxt][i] = jj;
        cur = nxt;
        if (!__syncthreads_or(jj >= 0)) break;
    }
    if (i < N) {
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint32_t *>(a.ws + L.mask_off) +
                                               ((size_t)b * N + i) * L.W4);
        for (int w = 0; w < L.W4; w += 4) {
            uint32_t x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = (w + k < W && i < n) ? anc[cur][i][w + k] : 0u;
            dst[w / 4] = make_uint4(x[0], x[1], x[2], x[3]);
        }
    }
}

// Plan. A query tile (b, kh, qt) needs T = ceil(P_b/128) prefix tiles plus
// the ceil(n_hi/128) tree tiles under its highest node. With
// tps = max(kMinTilesPerSplit, ceil(total / num_ctas)), it is cut into
// chunks of tps tiles plus one remainder chunk. Items are ordered longest
// first (counting sort on length) for the attention kernel's atomic queue,
// so the short remainders fill in behind the long chunks.
__device__ void plan(const Layout &L, const AttnArgs &a) {
    __shared__ int sh[32];
    __shared__ int hist[kHistBins];
    __shared__ int sP[kMaxBatch], sN[kMaxBatch];
    __shared__ int s_total;
    const int tid = threadIdx.x;
    for (int b = tid; b < L.B; b += blockDim.x) {
        const int P = a.prefix_lens[b], n = a.n_nodes[b];
        const bool ok = n >= 1 && n <= L.Nmax && P >= 0 && P <= L.Pcap;
        sP[b] = ok ? P : 0;
        sN[b] = ok ? n : 0;
    }
    for (int k = tid; k < kHistBins; k += blockDim.x) hist[k] = 0;
    __syncthreads();
    auto tiles = [&](int b, int qt) {
        const int n = sN[b], node0 = qt * L.NB;
        if (node0 >= n) return 0;
        return ceil_div(sP[b], kBN) + ceil_div(min(node0 + L.NB, n), kBN);
    };
    int local = 0;
    for (int k = tid; k < L.B * L.QT; k += blockDim.x) local += tiles(k / L.QT, k % L.QT);
    int excl;
    const int total = L.Hkv * block_exclusive_scan(local, &excl, sh);
    const int tps = max(kMinTilesPerSplit, ceil_div(total, max(1, a.num_ctas)));
    auto bin_of = [&](int size) { return min(size, kHistBins - 1); };

    QTile *qtab = reinterpret_cast<QTile *>(a.ws + L.qtab_off);
    Item *items = reinterpret_cast<Item *>(a.ws + L.items_off);
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + L.plan_off);
    // pass 1: split counts, length histogram, partial-slot bases
    int slot_run = 0;
    for (int base = 0; base < L.n_qtiles; base += blockDim.x) {
        const int q = base + tid;
        int ns = 0;
        if (q < L.n_qtiles) {
            const int T = tiles(q / (L.Hkv * L.QT), q % L.QT);
            ns = ceil_div(T, tps);
            for (int s = 0; s < ns; ++s) atomicAdd(&hist[bin_of(min(tps, T - s * tps))], 1);
        }
        int ex;
        const int tot = block_exclusive_scan(ns > 1 ? ns : 0, &ex, sh);
        if (q < L.n_qtiles) qtab[q] = QTile{ns, slot_run + ex, 0, 0};
        slot_run += tot;
    }
    __syncthreads();
    if (tid == 0) {   // longest first: starting offsets in descending length
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
        const int T = tiles(q / (L.Hkv * L.QT), q % L.QT);
        const int ns = ceil_div(T, tps);
        for (int s = 0; s < ns; ++s) {
            const int b0 = s * tps, b1 = min(T, b0 + tps);
            const int pos = atomicAdd(&hist[bin_of(b1 - b0)], 1);
            if (pos < L.max_items) items[pos] = Item{q, b0, b1, s};
        }
    }
    if (tid == 0) {
        // n_items <= n_qtiles + num_ctas = max_items always: sum ceil(T/tps)
        // <= total/tps + n_qtiles and tps >= total/num_ctas.
        *hdr = PlanHeader{min(s_total, L.max_items), 0, tps, total};
    }
}

__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(const Layout L, const AttnArgs a) {
    pdl_launch_dependents();
    if ((int)blockIdx.x < L.B)
        build_sequence(L, a, blockIdx.x);
    else
        plan(L, a);
}

}  // namespace

cudaError_t launch_tree_prep(const Layout &L, const AttnArgs &a, cudaStream_t s) {
    trace_begin("tree_prep", s);
    tree_prep_kernel<<<L.B + 1, kPrepThreads, 0, s>>>(L, a);
    cudaError_t e = cudaGetLastError();
    trace_end(s);
    return e;
}

}  // namespace jf
