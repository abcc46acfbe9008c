// jf_prep.cu - the kernel that runs before tree attention.
//
//  tree_prep_kernel  one block per sequence validates the tree and builds
//                    per-node ancestor bitmasks; one more block plans the
//                    attention kernel's stream-K split of the key tiles.
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

// Stream-K plan. Unit u (sequence b, KV head kh, query tile qt) needs
// T_u = ceil(P_b/128) prefix tiles plus the ceil(n_hi/128) tree tiles under
// its highest node. Concatenate all units' tiles (total) and give CTA c the
// equal range [c * total / C, (c + 1) * total / C), C = min(num_ctas,
// total / kMinTilesPerCta). A unit that several ranges cover is split; its
// split s is the s-th covering CTA (key order), writing partial slot
// slot_base + s for the combine kernel.
__device__ void plan(const Layout &L, const AttnArgs &a) {
    __shared__ int sh[32];
    __shared__ int sP[kMaxBatch], sN[kMaxBatch];
    const int tid = threadIdx.x;
    for (int b = tid; b < L.B; b += blockDim.x) {
        const int P = a.prefix_lens[b], n = a.n_nodes[b];
        const bool ok = n >= 1 && n <= L.Nmax && P >= 0 && P <= L.Pcap;
        sP[b] = ok ? P : 0;
        sN[b] = ok ? n : 0;
    }
    __syncthreads();
    auto tiles_of = [&](int u) {
        const int b = u / (L.Hkv * L.QT), qt = u % L.QT;
        const int n = sN[b], node0 = qt * L.NB;
        if (node0 >= n) return 0;
        return ceil_div(sP[b], kBN) + ceil_div(min(node0 + L.NB, n), kBN);
    };
    QTile *qtab = reinterpret_cast<QTile *>(a.ws + L.qtab_off);
    int32_t *cta_first = reinterpret_cast<int32_t *>(a.ws + L.first_off);
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(a.ws + L.plan_off);
    // pass 1: tile counts and their prefix sums
    int run = 0;
    for (int base = 0; base < L.n_qtiles; base += blockDim.x) {
        const int u = base + tid;
        const int T = u < L.n_qtiles ? tiles_of(u) : 0;
        int ex;
        const int tot = block_exclusive_scan(T, &ex, sh);
        if (u < L.n_qtiles) qtab[u] = QTile{0, 0, run + ex, T};
        run += tot;
    }
    const int total = run;
    const int C = max(1, min(a.num_ctas, total / kMinTilesPerCta));
    __syncthreads();   // qtab of every unit is visible to the whole block
    // pass 2: covering CTA ranges, split slots, each CTA's first unit
    int slot_run = 0;
    for (int base = 0; base < L.n_qtiles; base += blockDim.x) {
        const int u = base + tid;
        int ns = 0, S = 0, T = 0;
        if (u < L.n_qtiles) {
            S = qtab[u].tile_start;
            T = qtab[u].tiles;
            if (T > 0) {
                const int c_first = (int)(((long long)(S + 1) * C - 1) / total);
                const int c_last = (int)(((long long)(S + T) * C - 1) / total);
                ns = c_last - c_first + 1;
                for (int c = c_first; c <= c_last; ++c)   // ranges that start inside u
                    if ((long long)c * total / C >= S) cta_first[c] = u;
            }
        }
        int ex;
        const int tot = block_exclusive_scan(ns > 1 ? ns : 0, &ex, sh);
        if (u < L.n_qtiles) qtab[u] = QTile{ns, slot_run + ex, S, T};
        slot_run += tot;
    }
    if (tid == 0) *hdr = PlanHeader{total, total > 0 ? C : 0, 0, 0};
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
