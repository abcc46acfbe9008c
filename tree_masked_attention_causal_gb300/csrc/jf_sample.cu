// jf_sample.cu - stochastic tree verification on sm_103a.
//
// The paper's section 2.1 "Background" has the target verify the drafted
// tokens in parallel, citing Leviathan et al. (2023) for the rule. At a
// temperature T > 0 that rule is speculative sampling: a drafted token x
// drawn from the draft's distribution q is accepted with probability
// min(1, p(x) / q(x)), p the target's distribution; on rejection the
// target's residual max(p - q, 0), renormalised, takes p's place. In a
// tree it is applied at each accepted node u to u's children in index
// order, the residual carried from one rejected sibling to the next, and
// the walk moves to the first accepted child. When no child is accepted
// the next token is drawn from the final residual.
//
// After k rejections at u the residual is max(p - c_k q, 0) / N_k with
// c_0 = 0, N_0 = 1, c_{k+1} = c_k + N_k and N_k the mass of
// max(p - c_k q, 0): two scalars replace the residual vector, the
// acceptance ratio of token x is max(p(x) / q(x) - c_k, 0) / N_k, and
// each rejection costs one pass over the vocabulary for the new mass.
//
//  lse_chunk_kernel    HBM-bound scan of both logits arrays, chunked like
//                      the argmax (short chunks merged so that both arrays
//                      fit one wave): each CTA reduces its chunk of one row
//                      to (max z, sum 2^((z - max) log2(e) / T)).
//  sample_walk_kernel  a cluster of 16 CTAs per sequence (8 when the
//                      batch would not fit the SMs), launched
//                      programmatically after the scan. CTA 0 validates the
//                      tree, merges the row normalisers, walks the tree and
//                      takes every decision; each pass over the vocabulary
//                      (a residual mass, or the final Gumbel-max sample) is
//                      split over the other CTAs, which store their partial
//                      results into CTA 0 through distributed shared memory
//                      for it to combine in rank order. Those CTAs draw the
//                      Gumbel noise of their vocabulary slices into shared
//                      memory while CTA 0 gathers the tree, and then only
//                      run the commands CTA 0 posts, so every CTA meets the
//                      same sequence of cluster barriers.
//
// Random numbers: Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011) under key (seed, offset).
// Node c's acceptance uniform is word c % 4 of the block at counter
// (c / 4, b, 0, 0); vocabulary entry v's sampling uniform is word v % 4 at
// counter (v / 4, b, 1, 0). A word w gives (floor(w / 2^41) + 1/2) 2^-23.
// The sample is the v maximising ln r(v) - ln(-ln U(v)) over r(v) > 0,
// the lowest index on ties.
#include "jf_cluster.cuh"

namespace jf {
namespace {

constexpr int kSampleCluster = 8;     // CTAs sharing one sequence's vocabulary passes
constexpr int kSampleClusterBig = 16; // the same when the batch is small enough
constexpr int kSampleShortChunk = 16384;  // argmax chunks shorter than this are merged for the scan
constexpr size_t kSampleNoiseMax = 192 * 1024;  // dynamic shared memory for a slice's Gumbel noise
constexpr int kSampleThreads = 512;
constexpr int kSampleVecs = 4;        // 16-byte loads of each row in flight per thread

constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull, kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull, kPhiloxW1 = 0xBB67AE8584CAA73Bull;
constexpr float kLn2 = 0.69314718055994531f;

// Ten Philox4x64 rounds on counter c under key (k0, k1).
__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t hi0 = __umul64hi(kPhiloxM0, c[0]), lo0 = kPhiloxM0 * c[0];
        const uint64_t hi1 = __umul64hi(kPhiloxM1, c[2]), lo1 = kPhiloxM1 * c[2];
        const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
        k0 += kPhiloxW0;
        k1 += kPhiloxW1;
    }
}

// The 23-bit integer k of a word; the uniform is (k + 1/2) 2^-23, exact in fp32.
__device__ __forceinline__ uint32_t top23(uint64_t w) { return (uint32_t)(w >> 41); }
__device__ __forceinline__ float uniform_of(uint32_t k) { return ((float)k + 0.5f) * 0x1p-23f; }

// -ln(-ln U) for U = (k + 1/2) 2^-23: 1 - U = (2^23 - k - 1/2) 2^-23 is
// exact, so t = -ln U = -log1p(-(1 - U)) keeps full precision near U = 1;
// t lies in (6e-8, 16.7), where the fast natural log's error (about 1e-6
// absolute here) is far below the margins a sample's keys are told apart by.
__device__ __forceinline__ float gumbel_of(uint32_t k) {
    const float one_minus = ((float)(0x800000u - k) - 0.5f) * 0x1p-23f;
    return -__logf(-log1pf(-one_minus));
}

__device__ float accept_uniform(uint64_t seed, uint64_t offset, int b, int c) {
    uint64_t w[4] = {(uint64_t)(c >> 2), (uint64_t)(uint32_t)b, 0ull, 0ull};
    philox4x64_10(w, seed, offset);
    const int j = c & 3;
    const uint64_t x = j == 0 ? w[0] : j == 1 ? w[1] : j == 2 ? w[2] : w[3];
    return uniform_of(top23(x));
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&z)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        z[2 * j] = __uint_as_float(w[j] << 16);
        z[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float bf16_at(const __nv_bfloat16 *p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)) << 16);
}

// (m1, s1) and (m2, s2) are (max, sum 2^((z - max) k2)) of two sets; their union's.
__device__ __forceinline__ float2 lse_merge(float2 a, float2 b, float k2) {
    const float M = fmaxf(a.x, b.x);
    if (M == -__int_as_float(0x7f800000)) return make_float2(M, 0.f);
    return make_float2(M, a.y * ex2_approx((a.x - M) * k2) + b.y * ex2_approx((b.x - M) * k2));
}

__global__ void __launch_bounds__(kArgmaxThreads, kArgmaxCtasPerSm)
    lse_chunk_kernel(const __nv_bfloat16 *__restrict__ target, const __nv_bfloat16 *__restrict__ draft,
                     const int32_t *__restrict__ n_nodes, float2 *__restrict__ part, int Nmax, int V, int chunk,
                     int chunks, float k2) {
    // A programmatic dependent of the stream's previous kernel: nothing is
    // read before that grid has completed. Then the walk's clusters may
    // start: their work before their wait (the tree, the Gumbel noise)
    // overlaps this scan.
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    // Nodes from the last to the root, the sequences side by side and a
    // node's target and draft chunks together: the walks' passes mostly read
    // the rows of the roots and their first children, which are then the
    // last ones read and still in L2.
    const int nb = gridDim.y / Nmax;
    const int i = Nmax - 1 - (int)blockIdx.y / nb, b = (int)blockIdx.y - (Nmax - 1 - i) * nb;
    const int row = b * Nmax + i, which = blockIdx.x >= chunks ? 1 : 0;
    const int ch = blockIdx.x - which * chunks;
    const int tid = threadIdx.x;
    const int e0 = ch * chunk;
    const int nvec = (min(V, e0 + chunk) - e0) >> 3;         // V % 8 == 0
    const uint4 *src = reinterpret_cast<const uint4 *>((which ? draft : target) + (size_t)row * V + e0);
    // The first vectors go out before the row is known to be real (a
    // padding row's logits exist too): n_nodes's latency overlaps theirs.
    uint4 v[kArgmaxVecs];
#pragma unroll
    for (int u = 0; u < kArgmaxVecs; ++u) {
        const int k = tid + u * kArgmaxThreads;
        if (k < nvec) v[u] = ld_stream(src + k);
    }
    const int n = n_nodes[b];
    if (n < 1 || n > Nmax || i >= n) return;                 // padding row
    float2 acc = make_float2(-__int_as_float(0x7f800000), 0.f);
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
                float z[8];
                unpack8(v[u], z);
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
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, acc.x, o), __shfl_xor_sync(0xffffffffu, acc.y, o));
        acc = lse_merge(acc, other, k2);
    }
    __shared__ float2 sred[kArgmaxThreads / 32];
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) sred[warp] = acc;
    __syncthreads();
    if (tid == 0) {
        float2 t = sred[0];
        for (int w = 1; w < kArgmaxThreads / 32; ++w) t = lse_merge(t, sred[w], k2);
        const size_t rows = gridDim.y;
        part[((size_t)which * rows + row) * chunks + ch] = t;
    }
}

// ------------------------------------------------------------- the cluster

enum : int { kOpExit = 0, kOpMass = 1, kOpSample = 2 };

// A command CTA 0 posts to every CTA of its cluster: the pass and the row
// it runs over, with the residual's scale c and the row normalisers
// (max, log2 sum) of the target (p) and the draft (q).
struct Cmd {
    int op, row;
    float c, Mp, Lp, Mq, Lq, pad;
};

struct WalkShared {
    Cmd cmd;                     // this CTA's command (written by CTA 0)
    float part_f[kSampleClusterBig];   // CTA 0 only: each CTA's partial, stored there by that CTA:
    int part_i[kSampleClusterBig];     //   a residual mass, or the best Gumbel key and its index
    float red_f[kSampleThreads / 32];
    int red_i[kSampleThreads / 32];
    float bcast_f[2];
    int bcast_i[2];
    // CTA 0's copy of the tree, gathered before the scan completes: each
    // node's parent, first child and next sibling (index order, -1 when
    // none), its acceptance uniform, and the target and draft logits of
    // its token in its parent's rows (NaN for a token outside [0, V))
    int par[kMaxNodes], first_child[kMaxNodes], next_sib[kMaxNodes], path[kMaxNodes];
    uint32_t kids[kMaxNodes][8];
    float u[kMaxNodes], zp[kMaxNodes], zq[kMaxNodes];
    // per node row: (max, log2 sum) of the target and the draft
    float lse[kMaxNodes][4];
    // the walk's state, handed from thread 0 to the CTA
    int st_u, st_depth, st_next, st_op;
    float st_c, st_N;
};

// (a, ia) beats (b, ib): the larger key, then the lower index.
__device__ __forceinline__ bool beats(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia >= 0 && (ib < 0 || ia < ib));
}

// The vectors (8 entries each) of the vocabulary that cluster CTA `rank`
// covers: CTA 0 walks the tree and takes none; the others share them.
__device__ __forceinline__ void slice_of(int V, uint32_t rank, int &lo, int &hi) {
    const int nv = V >> 3, kw = (int)cluster_size() - 1;
    if (rank == 0) {
        lo = hi = 0;
        return;
    }
    lo = (int)((long long)(rank - 1) * nv / kw);
    hi = (int)((long long)rank * nv / kw);
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}

// Dynamic shared memory: the Gumbel noise of this CTA's vocabulary slice,
// when the launch gave it room (else the final pass draws it on the fly).
extern __shared__ float s_noise[];

__device__ __forceinline__ void philox_vec(int k, int b, uint64_t seed, uint64_t offset, uint64_t (&w)[8]) {
    uint64_t c0[4] = {(uint64_t)(2 * k), (uint64_t)(uint32_t)b, 1ull, 0ull};
    uint64_t c1[4] = {(uint64_t)(2 * k + 1), (uint64_t)(uint32_t)b, 1ull, 0ull};
    philox4x64_10(c0, seed, offset);
    philox4x64_10(c1, seed, offset);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        w[j] = c0[j];
        w[4 + j] = c1[j];
    }
}

// Before the scan completes: the noise of the slice into shared memory.
__device__ void precompute_noise(const SampleArgs &a, int V, int b, uint32_t rank) {
    int lo, hi;
    slice_of(V, rank, lo, hi);
    if ((uint32_t)(hi - lo) * 32u > dynamic_smem_bytes()) return;
    for (int k = lo + (int)threadIdx.x; k < hi; k += kSampleThreads) {
        uint64_t w[8];
        philox_vec(k, b, a.seed, a.offset, w);
#pragma unroll
        for (int j = 0; j < 8; ++j) s_noise[(k - lo) * 8 + j] = gumbel_of(top23(w[j]));
    }
}

// This CTA's share of a pass over row cmd.row: the residual mass of its
// vocabulary slice, or the best (key, index) of the Gumbel-max sample.
__device__ void run_slice(const Cmd &cmd, const SampleArgs &a, int V, int b, uint32_t rank, WalkShared &sh,
                          float &out_f, int &out_i) {
    const int tid = threadIdx.x;
    int lo, hi;
    slice_of(V, rank, lo, hi);
    const bool stored = (uint32_t)(hi - lo) * 32u <= dynamic_smem_bytes();
    const uint4 *rp = reinterpret_cast<const uint4 *>(a.target + (size_t)cmd.row * V);
    const uint4 *rq = reinterpret_cast<const uint4 *>(a.draft + (size_t)cmd.row * V);
    const float k2 = a.k2, c = cmd.c;
    const float Mp = cmd.Mp, Lp = cmd.Lp, Mq = cmd.Mq, Lq = cmd.Lq;
    float best = -__int_as_float(0x7f800000);
    int best_i = -1;
    float mass = 0.f;
    for (int k0 = lo + tid; k0 < hi; k0 += kSampleThreads * kSampleVecs) {
        uint4 vp[kSampleVecs], vq[kSampleVecs];
#pragma unroll
        for (int u = 0; u < kSampleVecs; ++u) {
            const int k = k0 + u * kSampleThreads;
            if (k < hi) {
                vp[u] = ld_stream(rp + k);
                if (c > 0.f) vq[u] = ld_stream(rq + k);
            }
        }
#pragma unroll 1
        for (int u = 0; u < kSampleVecs; ++u) {
            const int k = k0 + u * kSampleThreads;
            if (k >= hi) break;
            float zp[8], zq[8];
            unpack8(vp[u], zp);
            if (c > 0.f) unpack8(vq[u], zq);
            if (cmd.op == kOpMass) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float p = ex2_approx((zp[j] - Mp) * k2 - Lp);
                    const float q = ex2_approx((zq[j] - Mq) * k2 - Lq);
                    mass += fmaxf(p - c * q, 0.f);
                }
            } else {
                uint64_t w[8];
                if (!stored) philox_vec(k, b, a.seed, a.offset, w);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // log2 of p, then of the residual p - c q where it is positive
                    float lr = (zp[j] - Mp) * k2 - Lp;
                    bool keep = true;
                    if (c > 0.f) {
                        const float lq = (zq[j] - Mq) * k2 - Lq;
                        const float x = c * ex2_approx(lq - lr);
                        keep = x < 1.f;
                        lr += log1pf(-x) * 1.4426950408889634f;
                    }
                    if (keep) {
                        const float g = stored ? s_noise[(k - lo) * 8 + j] : gumbel_of(top23(w[j]));
                        const float key = lr * kLn2 + g;
                        if (key > best) {               // strictly: the first (lowest) index keeps a tie
                            best = key;
                            best_i = 8 * k + j;
                        }
                    }
                }
            }
        }
    }
    // block reduction in a fixed order
    const int warp = tid >> 5, lane = tid & 31;
    if (cmd.op == kOpMass) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mass += __shfl_xor_sync(0xffffffffu, mass, o);
        if (lane == 0) sh.red_f[warp] = mass;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w2 = 0; w2 < kSampleThreads / 32; ++w2) t += sh.red_f[w2];
            out_f = t;
            out_i = 0;
        }
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
            if (beats(ob, oi, best, best_i)) {
                best = ob;
                best_i = oi;
            }
        }
        if (lane == 0) {
            sh.red_f[warp] = best;
            sh.red_i[warp] = best_i;
        }
        __syncthreads();
        if (tid == 0) {
            float t = sh.red_f[0];
            int ti = sh.red_i[0];
            for (int w2 = 1; w2 < kSampleThreads / 32; ++w2)
                if (beats(sh.red_f[w2], sh.red_i[w2], t, ti)) {
                    t = sh.red_f[w2];
                    ti = sh.red_i[w2];
                }
            out_f = t;
            out_i = ti;
        }
    }
    __syncthreads();
}

// CTA 0 only: post a command to every CTA of the cluster (itself included).
__device__ void post(WalkShared &sh, int op, int row, float c, const float *lse) {
    const int tid = threadIdx.x;
    if (tid < (int)cluster_size()) {
        const uint32_t base = map_to_rank(smem_u32(&sh.cmd), tid);
        st_cluster(base + 0, (uint32_t)op);
        st_cluster(base + 4, (uint32_t)row);
        st_cluster(base + 8, __float_as_uint(c));
        for (int j = 0; j < 4; ++j) st_cluster(base + 12 + 4 * j, __float_as_uint(lse[j]));
    }
}

// CTA 0 only: one pass over row `row` split over the cluster. Returns the
// combined result (mass, or (key, index)) to every thread of CTA 0.
__device__ void cluster_pass(WalkShared &sh, const SampleArgs &a, int V, int b, int op, int row, float c,
                             const float *lse, float &res_f, int &res_i) {
    post(sh, op, row, c, lse);
    cluster_sync_all();                                      // commands visible
    if (threadIdx.x == 0) {                                  // CTA 0 has no slice of its own
        sh.part_f[0] = op == kOpMass ? 0.f : -__int_as_float(0x7f800000);
        sh.part_i[0] = -1;
    }
    cluster_sync_all();                                      // every partial is in place
    if (threadIdx.x == 0) {
        float t = op == kOpMass ? 0.f : -__int_as_float(0x7f800000);
        int ti = -1;
        const uint32_t kc = cluster_size();
        for (uint32_t r = 0; r < kc; ++r) {
            const float pf = sh.part_f[r];
            const int pi = sh.part_i[r];
            if (op == kOpMass) {
                t += pf;
            } else if (beats(pf, pi, t, ti)) {
                t = pf;
                ti = pi;
            }
        }
        sh.bcast_f[0] = t;
        sh.bcast_i[0] = ti;
    }
    __syncthreads();
    res_f = sh.bcast_f[0];
    res_i = sh.bcast_i[0];
    __syncthreads();
}

// The walk's states, as thread 0 hands them to the CTA.
enum : int { kWalkMass = 0, kWalkDone = 1 };

__global__ void __launch_bounds__(kSampleThreads, 2)
    sample_walk_kernel(const Layout L, const SampleArgs a, const float2 *__restrict__ part, int chunks,
                       int early) {
    if (early) pdl_launch_dependents();   // a follower may launch now; it waits for this grid before reading
    __shared__ WalkShared sh;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.y, tid = threadIdx.x;
    const int V = L.V, Nmax = L.Nmax, rows = L.B * L.Nmax;
    if (rank != 0) {
        // the cluster's workers: run each posted pass until told to stop
        precompute_noise(a, V, b, rank);
        pdl_wait_prior_grid();
        for (;;) {
            cluster_sync_all();                              // a command is posted
            const Cmd cmd = sh.cmd;                          // posted before the barrier
            if (cmd.op == kOpExit) break;
            float f = 0.f;
            int i = 0;
            run_slice(cmd, a, V, b, rank, sh, f, i);
            if (tid == 0) {                                  // into CTA 0's slot for this rank
                st_cluster(map_to_rank(smem_u32(&sh.part_f[rank]), 0), __float_as_uint(f));
                st_cluster(map_to_rank(smem_u32(&sh.part_i[rank]), 0), (uint32_t)i);
            }
            cluster_sync_all();                              // the partial is posted
        }
        return;
    }
    // CTA 0. Before the scan completes (inputs only): the tree, its child
    // lists, every node's acceptance uniform and its token's two logits.
    const int n = a.n_nodes[b];
    bool bad = n < 1 || n > Nmax;
    const size_t seq = (size_t)b * Nmax;
    if (!bad && tid < n) {
        const int p = a.parents[seq + tid];
        sh.par[tid] = p;
        bad = (tid == 0) ? (p != -1) : (p < 0 || p >= tid);
    }
    bad = __syncthreads_or(bad);
    if (!bad) {
        // children of each node as a bit set, then first child and next
        // sibling in index order from the set bits
        for (int k = tid; k < kMaxNodes * 8; k += kSampleThreads) (&sh.kids[0][0])[k] = 0u;
        __syncthreads();
        if (tid > 0 && tid < n) atomicOr(&sh.kids[sh.par[tid]][tid >> 5], 1u << (tid & 31));
        __syncthreads();
    }
    if (!bad && tid < n) {
        auto lowest_from = [&](const uint32_t *set, int from) {   // lowest member >= from, or -1
            for (int w = from >> 5; w < 8; ++w) {
                const uint32_t m = set[w] & (0xFFFFFFFFu << (w == (from >> 5) ? (from & 31) : 0));
                if (m) return 32 * w + __ffs(m) - 1;
            }
            return -1;
        };
        sh.first_child[tid] = lowest_from(sh.kids[tid], 0);
        sh.next_sib[tid] = tid > 0 && tid < kMaxNodes - 1 ? lowest_from(sh.kids[sh.par[tid]], tid + 1) : -1;
        float zp = __int_as_float(0x7fc00000), zq = zp;
        if (tid > 0) {
            const int x = a.tokens[seq + tid];
            if (x >= 0 && x < V) {
                const size_t at = (seq + sh.par[tid]) * (size_t)V + x;
                zp = bf16_at(a.target + at);
                zq = bf16_at(a.draft + at);
            }
            sh.u[tid] = accept_uniform(a.seed, a.offset, b, tid);
        }
        sh.zp[tid] = zp;
        sh.zq[tid] = zq;
    }
    pdl_wait_prior_grid();
    int32_t *path_out = a.accept_path + (size_t)b * (a.max_depth + 1);
    float lse[4] = {0.f, 0.f, 0.f, 0.f};
    if (bad) {
        for (int k = tid; k <= a.max_depth; k += kSampleThreads) path_out[k] = -1;
        if (tid == 0) {
            a.accept_len[b] = 0;
            a.next_token[b] = -1;
            set_status(a.status, JF_STATUS_BAD_TREE);
        }
        post(sh, kOpExit, 0, 0.f, lse);
        cluster_sync_all();
        return;
    }
    // every node row's normalisers, merged from the scan's chunks in chunk order
    for (int t = tid; t < 2 * n; t += kSampleThreads) {
        const int i = t >> 1, which = t & 1;
        const float2 *pr = part + ((size_t)which * rows + seq + i) * chunks;
        float2 acc = make_float2(-__int_as_float(0x7f800000), 0.f);
#pragma unroll 4
        for (int ch = 0; ch < chunks; ++ch) acc = lse_merge(acc, pr[ch], a.k2);
        sh.lse[i][2 * which] = acc.x;
        sh.lse[i][2 * which + 1] = log2f(acc.y);
    }
    if (tid == 0) {
        sh.st_u = 0;
        sh.st_depth = 0;
        sh.st_next = sh.first_child[0];
        sh.st_c = 0.f;
        sh.st_N = 1.f;
        sh.path[0] = 0;
    }
    __syncthreads();
    // Thread 0 walks the tree from shared memory until a rejection needs the
    // residual's new mass (a pass over the vocabulary by the whole cluster)
    // or the walk ends; the CTA then runs that pass and thread 0 goes on.
    for (;;) {
        if (tid == 0) {
            int u = sh.st_u, depth = sh.st_depth, ch = sh.st_next;
            float c = sh.st_c, N = sh.st_N;
            int op = kWalkDone;
            while (depth < a.max_depth && ch >= 0) {
                const float *ls = sh.lse[u];
                const float zp = sh.zp[ch], zq = sh.zq[ch];
                float ratio = 0.f;
                if (zp == zp) {                              // the token is in [0, V)
                    const float lp = (zp - ls[0]) * a.k2 - ls[1];
                    const float lq = (zq - ls[2]) * a.k2 - ls[3];
                    ratio = fmaxf(ex2_approx(lp - lq) - c, 0.f) / N;
                }
                if (sh.u[ch] < fminf(ratio, 1.f)) {          // accepted: go down
                    u = ch;
                    sh.path[++depth] = u;
                    ch = sh.first_child[u];
                    c = 0.f;
                    N = 1.f;
                    continue;
                }
                c += N;                                      // rejected: the residual needs its mass
                ch = sh.next_sib[ch];
                op = kWalkMass;
                break;
            }
            sh.st_u = u;
            sh.st_depth = depth;
            sh.st_next = ch;
            sh.st_c = c;
            sh.st_N = N;
            sh.st_op = op;
        }
        __syncthreads();
        const int op = sh.st_op, u = sh.st_u;
        for (int j = 0; j < 4; ++j) lse[j] = sh.lse[u][j];
        const float c = sh.st_c;
        __syncthreads();
        if (op == kWalkDone) break;
        float mass;
        int unused;
        cluster_pass(sh, a, V, b, kOpMass, (int)(seq + u), c, lse, mass, unused);
        if (tid == 0) {
            if (mass > 0.f) {
                sh.st_N = mass;
            } else {                                         // the residual vanished: sample from p
                sh.st_c = 0.f;
                sh.st_N = 1.f;
                sh.st_next = -1;
            }
        }
        __syncthreads();
    }
    const int u = sh.st_u, depth = sh.st_depth;
    float key;
    int token;
    cluster_pass(sh, a, V, b, kOpSample, (int)(seq + u), sh.st_c, lse, key, token);
    for (int k = tid; k <= a.max_depth; k += kSampleThreads) path_out[k] = k <= depth ? sh.path[k] : -1;
    if (tid == 0) {
        a.accept_len[b] = depth + 1;
        a.next_token[b] = token;
    }
    post(sh, kOpExit, 0, 0.f, lse);
    cluster_sync_all();
}

}  // namespace

cudaError_t launch_sample(const Layout &L, const SampleArgs &a, uint8_t *ws, int sms, cudaStream_t s) {
    const int rows = L.B * L.Nmax;
    float2 *part = reinterpret_cast<float2 *>(ws + L.lse_off);
    // The scan covers two arrays. With few rows the argmax's chunks are
    // short (a few thousand entries) and twice as many of them overrun one
    // wave: then the argmax's rule for twice the rows (one wave of
    // kArgmaxCtasPerSm CTAs per SM), never more chunks than the workspace
    // holds. Long chunks stay as the argmax cuts them (measured: one chunk
    // a row at the tree-256 shape, 0.84 of a wave, is slower than two).
    int per_row = L.chunks;
    if (L.V > 0 && rows > 0 && L.chunk < kSampleShortChunk) {
        per_row = 1;
        const long long rows2 = 2LL * rows;
        const long long fill = (4LL * sms + rows2 - 1) / rows2;
        const long long wave = (long long)kArgmaxCtasPerSm * sms / rows2;
        const long long want = fill < wave ? fill : wave;
        const long long most = L.chunks;
        if (want > per_row) per_row = (int)(want < most ? want : most);
    }
    const int chunk = L.V > 0 ? (int)align_up((size_t)ceil_div(L.V, per_row), kArgmaxGranule) : kArgmaxGranule;
    const int chunks = L.V > 0 ? ceil_div(L.V, chunk) : 1;
    trace_begin("lse_chunk", s);
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(2 * chunks, rows, 1);
    lc.blockDim = dim3(kArgmaxThreads, 1, 1);
    lc.stream = s;
    // With one or a few sequences the scan's launch overlaps the end of the
    // stream's previous kernel (a walk of an earlier call lets it start at
    // once). With a batch it does not: the scan's early CTAs then delayed
    // the batch's walks (serving batch +6.9 µs per call, one sequence -0.55).
    const int early = L.B * kSampleClusterBig <= sms ? 1 : 0;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = early;
    lc.attrs = la;
    lc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&lc, lse_chunk_kernel, a.target, a.draft, a.n_nodes, part, (int)L.Nmax,
                                       (int)L.V, chunk, chunks, a.k2);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(s);
    if (e != cudaSuccess) return e;
    trace_begin("sample_walk", s);
    // Once per device: the walk's shared-memory opt-in, then whether the
    // device schedules clusters of 16 of it (with that shared memory). 16
    // CTAs a sequence when it does and the batch leaves SMs for them, else 8
    // (the portable size).
    static int clusters_of[64] = {0};                    // 0: not yet asked; else 8 or 16
    static size_t whole_sm[64] = {0};                    // dynamic shared memory that fills a block's opt-in limit
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (clusters_of[dev] == 0) {
        cudaFuncAttributes fa{};
        int optin = 0;
        if (cudaFuncGetAttributes(&fa, sample_walk_kernel) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return cudaGetLastError();
        const size_t whole = (size_t)optin > fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
        whole_sm[dev] = whole > kSampleNoiseMax ? whole : kSampleNoiseMax;
        if (cudaFuncSetAttribute(sample_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)whole_sm[dev]) != cudaSuccess)
            return cudaGetLastError();
        int ok16 = 0;
        if (cudaFuncSetAttribute(sample_walk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
            cudaLaunchConfig_t probe{};
            probe.gridDim = dim3(kSampleClusterBig, 1, 1);
            probe.blockDim = dim3(kSampleThreads, 1, 1);
            probe.dynamicSmemBytes = kSampleNoiseMax;
            cudaLaunchAttribute ca[1];
            ca[0].id = cudaLaunchAttributeClusterDimension;
            ca[0].val.clusterDim.x = kSampleClusterBig;
            ca[0].val.clusterDim.y = 1;
            ca[0].val.clusterDim.z = 1;
            probe.attrs = ca;
            probe.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, sample_walk_kernel, &probe) == cudaSuccess && clusters > 0)
                ok16 = 1;
        }
        // and whether clusters of 8 fit with a whole block's shared memory each
        {
            cudaLaunchConfig_t probe{};
            probe.gridDim = dim3(kSampleCluster, 1, 1);
            probe.blockDim = dim3(kSampleThreads, 1, 1);
            probe.dynamicSmemBytes = whole_sm[dev];
            cudaLaunchAttribute ca[1];
            ca[0].id = cudaLaunchAttributeClusterDimension;
            ca[0].val.clusterDim.x = kSampleCluster;
            ca[0].val.clusterDim.y = 1;
            ca[0].val.clusterDim.z = 1;
            probe.attrs = ca;
            probe.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, sample_walk_kernel, &probe) != cudaSuccess || clusters < 1)
                whole_sm[dev] = 0;
        }
        cudaGetLastError();                                  // a refused query leaves no error behind
        clusters_of[dev] = ok16 ? kSampleClusterBig : kSampleCluster;
    }
    const int kc = (clusters_of[dev] == kSampleClusterBig && L.B * kSampleClusterBig <= sms) ? kSampleClusterBig
                                                                                            : kSampleCluster;
    // room for the Gumbel noise of one worker CTA's vocabulary slice, if it fits
    const size_t noise = (size_t)((L.V / 8 + kc - 2) / (kc - 1)) * 32;
    size_t dyn = noise <= kSampleNoiseMax ? noise : 0;
    // With a cluster a sequence on most SMs (a batch), a walk CTA resident
    // beside scan CTAs holds their share of the SM through the rest of the
    // scan, which costs more than its early start gains (serving batch:
    // 159 -> 148 µs per call). Asking for all the shared memory a block may
    // have keeps it off every SM that still runs a scan CTA: the clusters
    // start on SMs as the scan leaves them, their pre-wait work overlapping
    // the scan's tail. A few clusters (one sequence) start at once; more
    // than one wave of them at one CTA per SM keep two CTAs per SM.
    if (L.B * kSampleClusterBig > sms && L.B * kc <= sms && noise <= whole_sm[dev]) dyn = whole_sm[dev];
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(kc, L.B, 1);
    cfg.blockDim = dim3(kSampleThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, sample_walk_kernel, L, a, static_cast<const float2 *>(part), chunks, early);
    trace_end(s);
    return e;
}

}  // namespace jf
