// jf_common.cuh - shared definitions of the sm_103a kernels: tile sizes, the
// workspace layout, and inline-PTX wrappers for mbarrier, TMA (cp.async.bulk
// .tensor) and the 5th-generation tensor core (tcgen05 + TMEM).
//
// The PTX wrappers follow the PTX ISA's descriptions of these instructions.
// Every wait on an mbarrier is bounded: after kTimeoutNs it sets
// JF_STATUS_TIMEOUT, raises the CTA's abort flag and returns false, so no
// kernel can spin forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/jf_tree.h"

namespace jf {

// ---------------------------------------------------------------- tiling
constexpr int kBM = 128;          // rows of one tcgen05 MMA tile (= TMEM lanes)
constexpr int kRows = 128;        // stacked query rows per work unit (one MMA tile)
constexpr int kBN = 128;          // keys per KV tile (the plan divides by it with >> 7)
constexpr int kMaxNodes = 256;    // tree slots per sequence
constexpr int kMaxCtas = 256;     // cap on the persistent attention grid
constexpr int kMinTilesPerCta = 2;   // smallest key range a CTA is given
constexpr int kMaxBatch = 1024;   // sequences per jf_tree_attention call
constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxVecs = 8;    // 16-byte loads in flight per thread
constexpr int kArgmaxCtasPerSm = 4;  // resident argmax CTAs per SM (64 registers: no spills)
constexpr int kArgmaxMaxChunk = 76800;  // target bf16 of one logits row per CTA (150 KB)
constexpr int kArgmaxGranule = kArgmaxThreads * 8;  // chunks are whole vectors per thread
constexpr int kScoreMaxK = 16;    // top-k of the path scoring, at most
constexpr int kMaxSms = 256;      // SM count the workspace is sized for (the chunking uses the real one)
// The limit of one wait. A test build shortens it (JF_WAIT_NS) to make a
// wait run out; the drains at exit keep their own, longer limit.
#ifndef JF_WAIT_NS
#define JF_WAIT_NS 2000000000ull
#endif
constexpr unsigned long long kTimeoutNs = JF_WAIT_NS;             // 2 s per wait
constexpr unsigned long long kDrainTimeoutNs = 250000000ull;      // 250 ms for a drain at exit

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Per work unit (kRows stacked query rows of one sequence and KV head),
// written by the attention CTA whose key range holds the unit's first tile
// and read by the combine kernel: how many CTA ranges split the unit, the
// first of them, and whether the unit is that CTA's first item.
struct QTile {
    int32_t n_splits;    // CTA ranges covering the unit (1 = not split)
    int32_t c_first;     // CTA whose range holds the unit's first tile
    int32_t first_item;  // 1 if the unit starts that CTA's range
    int32_t tile_start;  // the unit's first tile in the concatenation of all units' tiles
};

// Byte offsets of the workspace regions. Attention regions come first, then
// the verify region; the two never overlap.
struct Layout {
    int32_t B, Nmax, Hq, Hkv, G, D, Pcap, V;
    int32_t QT;          // work units per (sequence, kv head)
    int32_t NB;          // nodes per work unit = kRows / G
    int32_t lgG, lgNB;   // log2 of G and NB (both powers of two)
    int32_t n_qtiles;    // work units: B * Hkv * QT
    int32_t max_pieces;  // partial slots: two per CTA (its first and its last item)
    int32_t chunk;       // bf16 elements of a logits row per argmax CTA
    int32_t chunks;      // argmax chunks per logits row
    size_t qtab_off, ml_off, opart_off;
    size_t amp_off;
    size_t lse_off;      // stochastic verify: (max, sum) per (target | draft, row, chunk);
                         // path scoring: (max, log2 sum) per row
    size_t total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The layout depends only on the shape (never on prefix lengths or trees).
// `sms` is the SM count the argmax chunking is cut for: the device's own in
// a call, kMaxSms when sizing a workspace (more SMs never mean fewer
// chunks, so a call's layout always fits the sized one).
inline Layout make_layout(int B, int Nmax, int Hq, int Hkv, int D, int Pcap, int V, int sms) {
    Layout L{};
    L.B = B; L.Nmax = Nmax; L.Hq = Hq; L.Hkv = Hkv; L.G = Hq / Hkv; L.D = D; L.Pcap = Pcap; L.V = V;
    L.NB = kRows / L.G;
    L.lgG = 0;
    while ((1 << L.lgG) < L.G) ++L.lgG;
    L.lgNB = 7 - L.lgG;   // kRows = 128
    L.QT = ceil_div(Nmax, L.NB);
    L.n_qtiles = B * Hkv * L.QT;
    L.max_pieces = 2 * kMaxCtas;
    // Argmax chunks: rows are cut into pieces of about kArgmaxMaxChunk; with
    // few rows into more, so that the grid reaches ~4 CTAs per SM while it
    // still fits one wave of kArgmaxCtasPerSm per SM.
    int per_row = V > 0 ? ceil_div(V, kArgmaxMaxChunk) : 1;
    const long long rows = (long long)B * Nmax;
    if (V > 0 && rows > 0) {
        const long long fill = (4LL * sms + rows - 1) / rows;
        const long long wave = (long long)kArgmaxCtasPerSm * sms / rows;
        const long long want = fill < wave ? fill : wave;
        const long long most = ceil_div(V, kArgmaxGranule);
        if (want > per_row) per_row = (int)(want < most ? want : most);
    }
    L.chunk = V > 0 ? (int)align_up((size_t)ceil_div(V, per_row), kArgmaxGranule) : kArgmaxGranule;
    L.chunks = V > 0 ? ceil_div(V, L.chunk) : 1;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    L.qtab_off = take(sizeof(QTile) * (size_t)L.n_qtiles);
    L.ml_off = take(sizeof(float4) * (size_t)L.max_pieces * kRows);   // (m, l, e0, e1)
    L.opart_off = take(2 * (size_t)L.max_pieces * kRows * D);   // fp16 rows, divided by l, scaled by 2^-e per half
    L.amp_off = take(sizeof(int2) * (size_t)B * Nmax * L.chunks);
    L.lse_off = take(2 * sizeof(float2) * (size_t)B * Nmax * L.chunks);
    L.total = off;
    return L;
}

// ------------------------------------------------------------- the plan
// Work unit u = (b, kh, qt), u = (b * Hkv + kh) * QT + qt, holds kRows
// stacked query rows: the G query heads of KV head kh for nodes
// qt * NB .. qt * NB + NB - 1 of sequence b. Its keys are ceil(P / 128)
// prefix tiles followed by the tree tiles up to its highest node (with
// parents[i] < i no key above a node can be its ancestor). The units' tiles
// are concatenated in u order and CTA c of C takes the equal range
// [c * total / C, (c + 1) * total / C) (stream-K). Every kernel derives this
// plan from prefix_lens and n_nodes alone, with the functions below.

// A sequence with an out-of-range length or prefix gets no work.
__host__ __device__ inline bool seq_valid(int P, int n, const Layout &L) {
    return n >= 1 && n <= L.Nmax && P >= 0 && P <= L.Pcap;
}

__device__ __forceinline__ int unit_tiles(int P, int n, int qt, const Layout &L) {
    const int node0 = qt << L.lgNB;
    if (node0 >= n) return 0;
    return ((P + kBN - 1) >> 7) + ((min(node0 + L.NB, n) + kBN - 1) >> 7);
}

// Tiles of all units of one KV head of a valid sequence, in closed form:
// unit qt < nq - 1 reaches node (qt + 1) * NB, i.e. ceil((qt + 1) / G) tree
// tiles since NB * G = 128, and the last unit reaches node n.
__device__ __forceinline__ int head_tiles(int P, int n, const Layout &L) {
    const int nq = (n + L.NB - 1) >> L.lgNB;
    const int m = nq - 1, q = m >> L.lgG, r = m - (q << L.lgG);
    return nq * ((P + kBN - 1) >> 7) + ((q * (q + 1) / 2) << L.lgG) + r * (q + 1) + ((n + kBN - 1) >> 7);
}

__device__ __forceinline__ int plan_ctas(int total, int num_ctas) {
    return max(1, min(num_ctas, total / kMinTilesPerCta));
}

// First tile of CTA c's range, floor(c * total / C), in 32-bit arithmetic:
// with total = C * qt + rt, it is c * qt + floor(c * rt / C) (c, rt < 256).
__device__ __forceinline__ int range_start(int c, int qt, int rt, int C) { return c * qt + (c * rt) / C; }

// Warp-collective: the CTA whose range holds tile x, i.e. the number of
// CTAs c >= 1 whose range starts at or before x.
__device__ __forceinline__ int cta_of_tile(int x, int qt, int rt, int C) {
    const int lane = threadIdx.x & 31;
    int n = 0;
#pragma unroll 1
    for (int c0 = 1; c0 < C; c0 += 32) {
        const int c = c0 + lane;
        n += __popc(__ballot_sync(0xffffffffu, c < C && range_start(c, qt, rt, C) <= x));
    }
    return n;
}

// Warp-collective: the plan as seen from CTA c. Returns total tiles and C,
// and, if the CTA's range [lo, hi) is not empty, the sequence b holding
// tile lo with its first tile, prefix length and node count (every lane gets
// the same). One pass over the sequences; a batch of up to 32 sequences is
// read from memory once.
// The split is weighted: every unit with work is preceded by alpha virtual
// tiles, and the virtual sequence is cut into C equal ranges. A CTA whose
// range crosses into another unit (an extra epilogue and pipeline refill)
// thus gets about alpha fewer real tiles. alpha = min(kSwitchTiles, half of
// the real tiles per CTA), so that no range can hold virtual tiles only.
constexpr int kSwitchTiles = 4;

struct PlanSeq {
    int n_ctas, alpha;
    int qt, rt;         // virtual total = n_ctas * qt + rt
    int lo, hi;         // this CTA's virtual range
    int b, P, n;        // the sequence holding virtual tile lo
    int seq_start;      // its first virtual tile
    int kv_tiles;       // prefix tiles of all KV heads of all valid sequences
};

// Units with work in one KV head of a valid sequence.
__device__ __forceinline__ int head_units(int n, const Layout &L) { return (n + L.NB - 1) >> L.lgNB; }

// Warp-collective: the plan as seen from CTA c (every lane gets the same).
// One pass over the sequences; a batch of up to 32 sequences is read from
// memory once.
__device__ inline PlanSeq plan_locate(const Layout &L, const int32_t *prefix_lens, const int32_t *n_nodes, int c,
                                      int num_ctas) {
    const int lane = threadIdx.x & 31;
    PlanSeq r{};
    r.b = -1;
    int P0 = 0, n0 = 0;                              // this lane's sequence of the first 32
    int tiles = 0, units = 0, kv = 0;
#pragma unroll 1
    for (int b0 = 0; b0 < L.B; b0 += 32) {
        const int b = b0 + lane;
        int P = 0, n = 0;
        if (b < L.B) {
            P = prefix_lens[b];
            n = n_nodes[b];
        }
        if (b0 == 0) {
            P0 = P;
            n0 = n;
        }
        if (b < L.B && seq_valid(P, n, L)) {
            tiles += L.Hkv * head_tiles(P, n, L);
            units += L.Hkv * head_units(n, L);
            kv += L.Hkv * ((P + kBN - 1) >> 7);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
        units += __shfl_xor_sync(0xffffffffu, units, o);
        kv += __shfl_xor_sync(0xffffffffu, kv, o);
    }
    r.kv_tiles = kv;
    r.n_ctas = tiles > 0 ? plan_ctas(tiles, num_ctas) : 0;
    if (c >= r.n_ctas) return r;
    r.alpha = min(kSwitchTiles, tiles / r.n_ctas / 2);
    const int total_v = tiles + r.alpha * units;
    r.qt = total_v / r.n_ctas;
    r.rt = total_v - r.qt * r.n_ctas;
    r.lo = range_start(c, r.qt, r.rt, r.n_ctas);
    r.hi = range_start(c + 1, r.qt, r.rt, r.n_ctas);
    int carry = 0;
#pragma unroll 1
    for (int b0 = 0; b0 < L.B; b0 += 32) {
        const int b = b0 + lane;
        int P = P0, n = n0;
        if (b0 > 0) {
            P = b < L.B ? prefix_lens[b] : 0;
            n = b < L.B ? n_nodes[b] : 0;
        }
        const int t = (b < L.B && seq_valid(P, n, L))
                          ? L.Hkv * (head_tiles(P, n, L) + r.alpha * head_units(n, L)) : 0;
        int incl = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int start = carry + incl - t;
        const unsigned hit = __ballot_sync(0xffffffffu, t > 0 && r.lo >= start && r.lo < start + t);
        if (hit) {
            const int src = __ffs(hit) - 1;
            r.b = b0 + src;
            r.seq_start = __shfl_sync(0xffffffffu, start, src);
            r.P = __shfl_sync(0xffffffffu, P, src);
            r.n = __shfl_sync(0xffffffffu, n, src);
            return r;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    return r;
}

// ------------------------------------------------------------- PTX: misc
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t flag) {
    if (status) atomicOr(status, flag);
}

// ------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete. Returns false
// (and raises *abort) if the CTA aborted or the wait ran past kTimeoutNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > kTimeoutNs) {
            *abort = 1;
            set_status(status, JF_STATUS_TIMEOUT);
            return false;
        }
    }
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 3-D tiled bulk tensor load global -> shared, completing on `bar`.
// Coordinates are element indices, innermost first.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 3-D tiled bulk tensor store shared -> global (bulk async-group completion).
// Coordinates are element indices, innermost first; none may be negative.
__device__ __forceinline__ void tma_store_3d(const void *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has read its shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bring the line holding p into L2 (no register result). L2 is coherent, so
// this is safe even before a programmatic wait on the line's producer.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Bring the line holding p into L1 (no register result).
__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Generic-proxy shared-memory writes -> visible to the async proxy (TMA/MMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------- tcgen05 and TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family layout:
// start>>4 in bits 0-13, leading byte offset>>4 in 16-29, stride byte
// offset>>4 in 32-45, descriptor version 1 in 46-47, swizzle mode 2 =
// 128B in 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulate:
// D format bits 4-5 (1 = f32), A format 7-9 and B format 10-12 (1 = bf16),
// A/B major bits 15/16 (0 = K-major, 1 = MN-major), N>>3 in 17-22,
// M>>4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one CTA. Called by a whole converged
// warp with warp-uniform operands; one elected lane issues. Issued this way,
// back to back, one warp keeps the tensor core at its full rate (64 cycles
// per 128 x 128 x 16); from a single-lane branch an MMA costs 110-150 cycles
// (measured on GB300).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], one CTA; warp-collective like mma_ss.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the elected lane issued
// so far has completed. Warp-collective like mma_ss.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

#define JF_R8(i) "=r"(v[i + 0]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), \
                 "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
#define JF_W8(i) "r"(v[i + 0]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), \
                 "r"(v[i + 4]), "r"(v[i + 5]), "r"(v[i + 6]), "r"(v[i + 7])

// Load 32 consecutive fp32 columns of this thread's TMEM lane (32x32b
// shape: warp w of a warpgroup reads lanes 32w..32w+31) and wait for them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : JF_R8(0), JF_R8(8), JF_R8(16), JF_R8(24)
        : "r"(taddr)
        : "memory");
}

// Store 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        JF_W8(0), JF_W8(8), JF_W8(16), JF_W8(24)
        : "memory");
}

// Store 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef JF_R8
#undef JF_W8

// Load 128 consecutive fp32 columns of this thread's TMEM lane and wait for
// them in the same statement (so no use can be scheduled before the wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&v)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63]), "=r"(v[64]), "=r"(v[65]), "=r"(v[66]), "=r"(v[67]), "=r"(v[68]), "=r"(v[69]), "=r"(v[70]), "=r"(v[71]), "=r"(v[72]), "=r"(v[73]), "=r"(v[74]), "=r"(v[75]), "=r"(v[76]), "=r"(v[77]), "=r"(v[78]), "=r"(v[79]), "=r"(v[80]), "=r"(v[81]), "=r"(v[82]), "=r"(v[83]), "=r"(v[84]), "=r"(v[85]), "=r"(v[86]), "=r"(v[87]), "=r"(v[88]), "=r"(v[89]), "=r"(v[90]), "=r"(v[91]), "=r"(v[92]), "=r"(v[93]), "=r"(v[94]), "=r"(v[95]), "=r"(v[96]), "=r"(v[97]), "=r"(v[98]), "=r"(v[99]), "=r"(v[100]), "=r"(v[101]), "=r"(v[102]), "=r"(v[103]), "=r"(v[104]), "=r"(v[105]), "=r"(v[106]), "=r"(v[107]), "=r"(v[108]), "=r"(v[109]), "=r"(v[110]), "=r"(v[111]), "=r"(v[112]), "=r"(v[113]), "=r"(v[114]), "=r"(v[115]), "=r"(v[116]), "=r"(v[117]), "=r"(v[118]), "=r"(v[119]), "=r"(v[120]), "=r"(v[121]), "=r"(v[122]), "=r"(v[123]), "=r"(v[124]), "=r"(v[125]), "=r"(v[126]), "=r"(v[127])
        : "r"(taddr)
        : "memory");
}

// Load 64 consecutive fp32 columns of this thread's TMEM lane (+ wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
        : "r"(taddr)
        : "memory");
}

// Per-warpgroup register budget (all 128 threads of the warpgroup execute
// it). The launch's total (threads x registers per thread) is the pool.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Store 64 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait here until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 values in one 64-bit register, for the packed f32x2 arithmetic of
// sm_100 and later (one instruction per pair of lanes' values).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f32x2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x (low half) = lo
    return *reinterpret_cast<uint32_t *>(&h);
}

// ------------------------------------------------------ kernel launchers
// (defined in the .cu files, called by the C ABI in jf_api.cu)
struct AttnMaps {
    CUtensorMap q, k_cache, v_cache, tree_k, tree_v;
    CUtensorMap out;    // bf16 [B * Nmax, Hq, d], box {64, G, NB}: one work unit, like q
    CUtensorMap part;   // fp16 [pieces, 128 rows, d], box {64, 128, 1}: split partials
};

struct AttnArgs {
    const int32_t *prefix_lens;
    const int32_t *parents;
    const int32_t *n_nodes;
    __nv_bfloat16 *out;
    uint8_t *ws;
    int32_t *status;
    float scale_log2;
    int32_t num_ctas;    // persistent grid size of the attention kernel
    // Paged prefix cache (page_lg >= 0): page j of sequence b is physical
    // page block_table[b * pages_per_seq + j] of a [num_pages, 2^page_lg,
    // Hkv, d] array; the k_cache / v_cache maps then cover that array.
    const int32_t *block_table;
    int32_t page_lg;     // log2 of the page size, -1 for the contiguous cache
    int32_t pages_per_seq;
    int32_t num_pages;
};

cudaError_t launch_tree_attention(const Layout &L, const AttnMaps &m, const AttnArgs &a,
                                  cudaStream_t s);
cudaError_t launch_split_combine(const Layout &L, const AttnArgs &a, cudaStream_t s);
// Paged when page_lg >= 0: the caches are [num_pages, 2^page_lg, Hkv, d] pools.
cudaError_t launch_commit_kv(const Layout &L, const __nv_bfloat16 *tree_k, const __nv_bfloat16 *tree_v,
                             const int32_t *n_nodes, const int32_t *accept_len, const int32_t *accept_path,
                             __nv_bfloat16 *k_cache, __nv_bfloat16 *v_cache, int32_t *prefix_lens, int32_t max_depth,
                             int32_t *status, cudaStream_t s, const int32_t *block_table = nullptr,
                             int32_t page_lg = -1, int32_t num_pages = 0);
cudaError_t launch_argmax(const Layout &L, const __nv_bfloat16 *logits, const int32_t *n_nodes,
                          uint8_t *ws, cudaStream_t s);
cudaError_t launch_accept_walk(const Layout &L, const int32_t *tokens, const int32_t *parents,
                               const int32_t *n_nodes, int32_t *accept_len, int32_t *accept_path,
                               int32_t *argmax_out, int32_t max_depth, uint8_t *ws, int32_t *status,
                               cudaStream_t s);

// Stochastic verification (jf_sample.cu): the per-row normalisers of the
// target and draft logits, then the walk and the final sample.
struct SampleArgs {
    const __nv_bfloat16 *target, *draft;
    const int32_t *tokens, *parents, *n_nodes;
    int32_t *accept_len, *accept_path, *next_token, *status;
    float k2;                 // log2(e) / temperature
    uint64_t seed, offset;    // Philox key
    int32_t max_depth;
};
cudaError_t launch_sample(const Layout &L, const SampleArgs &a, uint8_t *ws, int sms, cudaStream_t s);

// Draft-side path scoring (jf_score.cu).
struct ScoreArgs {
    const __nv_bfloat16 *draft;
    const int32_t *tokens, *parents, *n_nodes;
    float *node_lp, *path_lp, *topk_lp, *cand_score;
    int32_t *topk_token, *cand_parent, *cand_token, *status;
    float k2;                 // log2(e) / temperature
    int32_t top_k, budget;
};
cudaError_t launch_score(const Layout &L, const ScoreArgs &a, uint8_t *ws, int sms, cudaStream_t s);

// Host-side launch bookkeeping (jf_api.cu): counts launches and records the
// armed trace events around each one.
void trace_begin(const char *name, cudaStream_t s);
void trace_end(cudaStream_t s);

}  // namespace jf
