// jf_attn.cu - tree-causal attention forward on sm_103a (TMA + tcgen05/TMEM).
//
// What it computes ("JetFlow: Scaling Speculative Decoding with Parallel Tree
// Drafting", blog, section "What JetFlow Does Differently"): all tree nodes in
// one pass; node i attends to every prefix key and to the tree keys of its
// ancestors and itself, never to siblings or descendants.
//
// Design
//  * Query stacking (GQA). The G = Hq/Hkv query heads that share a KV head
//    are stacked with the nodes into a work unit of 128 rows (one tcgen05
//    MMA tile): row r = node_local * G + g. One 3-D TMA box
//    {64 d, G heads, 128/G nodes} loads the unit straight from
//    q[B, Nmax, Hq, d]. Each K/V tile in shared memory then serves all G
//    heads.
//  * Virtual key sequence. Per unit, the keys are ceil(P/128) prefix tiles
//    (from k_cache/v_cache) followed by ceil(n_hi/128) dense tree tiles (from
//    tree_k/tree_v). Here n_hi is one past the unit's highest node, and
//    parents[i] < i means no key above a node is ever its ancestor. The
//    ancestor bits of a tree tile come from a walk up the parents array and
//    mask the tile in registers; a key-count bound masks the ragged last
//    prefix tile.
//  * Stream-K split of the keys. Each CTA derives the plan itself from
//    prefix_lens and n_nodes: every unit's key tiles concatenated, and an
//    equal contiguous range per CTA. A CTA walks its range as one or a few
//    items (one per unit it touches). A unit covered by a single range is
//    normalised and written as bf16 here. Every piece of a unit covered by
//    several ranges writes its rows O / l as fp16, scaled by 2^-e per half
//    row, with (m, l, e) in fp32 beside them, which the combine kernel
//    merges; the CTA where a unit starts records the unit's split plan.
//  * One CTA per SM, 12 warps:
//      warps 0-7  softmax: warp w owns TMEM lanes 32 (w % 4).. (rows) for
//                 the key tiles g with g % 2 == w / 4; the two warps of a
//                 row quadrant alternate tiles and hide each other's
//                 latencies
//      warp 8     TMA producer of Q (per item, double-buffered) and of the
//                 NK-stage K ring
//      warp 11    TMA producer of the NV-stage V ring
//      warp 9     QK^T issuer and TMEM owner: S(g) = Q K(g)^T into S buffer g % 3
//      warp 10    PV issuer: O += P(g) V(g)
//    MMAs are issued by a whole converged warp (elected lane, warp-uniform
//    operands); unrolled back to back, one warp keeps the tensor core at its
//    full rate. The two issuers run concurrently on independent
//    accumulators.
//    TMEM: S buffers at columns 0, 128, 256; O at [384, 384+d). P is written
//    back as bf16 over the first 64 columns of its own S. The three S buffers
//    are a ring between the two issuers: QK^T may run two tiles ahead of the
//    softmax, and a buffer returns to the QK issuer when the PV that read its
//    P completes.
//  * Softmax per tile (one warp per row quadrant): one 128-column TMEM load
//    for the row max, the running max handed over from the previous tile's
//    owner, then ex2 on the MUFU pipe, bf16 packing and the P store in a
//    rolled loop over 64-column chunks read again from TMEM; the scaling
//    and the row sums use packed f32x2 arithmetic. Instruction fetch is a
//    first-order cost for this kernel, so the hot loop is kept small.
//  * Online softmax in the exp2 domain, lazy rescale: O is rescaled only
//    when a row max grows by more than 2^8, by the owner of that tile, once
//    the previous tile's PV has completed. The first PV of an item waits
//    until every softmax warp has read the previous item's O.
//  * Launched as a programmatic dependent of the previous kernel: barrier
//    set-up, the TMEM allocation and the tensor-map prefetches run before
//    the wait, every input read after it. No kernel of its own runs before
//    it. Tree validation and the NaN rows of malformed sequences are left
//    to the combine kernel, which overwrites whatever this kernel wrote for
//    them.
//  * Rows of padding nodes are computed but never stored. V rows past the
//    prefix length or past n_nodes are zeroed in shared memory before the
//    PV MMA, so NaN in unused cache rows cannot reach an output.
#include "jf_common.cuh"

namespace jf {
namespace {

struct ItemInfo {
    int32_t valid, b, kh, qt, tb, te, t_pre, P, n, ns, slot, qtile, rot, pad1, pad2, pad3;
};

constexpr long long kRotateBytes = 64ll << 20;         // half the L2

// The prefix tile that tile t (< t_pre) of an item stands for. When the
// prefix K/V of the call exceed half the L2, a unit walks its prefix tiles
// from `rot` on and wraps around, `rot` chosen so that the first range
// boundary inside the unit falls on prefix tile 0. The pieces of the units
// of one KV head then begin on the same few prefix tiles and move through
// them side by side, so that L2 serves a tile to all of them after one DRAM
// read instead of evicting it between their visits. (When the K/V fit in
// L2 every tile is read from DRAM once anyway, and the rotation measured
// slightly slower.) The online softmax does not depend on the order.
__device__ __forceinline__ int prefix_tile(const ItemInfo &info, int t) {
    const int p = t + info.rot;
    return p >= info.t_pre ? p - info.t_pre : p;
}

template <int D>
struct AttnCfg {
    static constexpr int NQ = 2;                            // Q buffers: the next unit's Q loads early
    static constexpr int NK = D == 128 ? 3 : 4;             // K ring stages (released right after QK^T)
    static constexpr int NV = D == 128 ? 2 : 6;             // V ring stages
    static constexpr int NS = 3;                            // S/P buffers in TMEM
    static constexpr int kBoxes = D / 64;                   // 64-column (128-byte) swizzled boxes
    static constexpr uint32_t kQBoxBytes = kRows * 128;     // one box: 128 rows x 128 B
    static constexpr uint32_t kQBytes = kRows * D * 2;
    static constexpr uint32_t kTileBytes = kBN * D * 2;
    static constexpr uint32_t q_off = 0;
    static constexpr uint32_t k_off = q_off + NQ * kQBytes;
    static constexpr uint32_t v_off = k_off + NK * kTileBytes;
    static constexpr uint32_t bar_off = v_off + NV * kTileBytes;
    static constexpr int B_Q_FULL = 0, B_Q_EMPTY = B_Q_FULL + NQ, B_K_FULL = B_Q_EMPTY + NQ, B_K_EMPTY = B_K_FULL + NK,
                         B_V_FULL = B_K_EMPTY + NK, B_V_EMPTY = B_V_FULL + NV, B_S_FULL = B_V_EMPTY + NV,
                         B_S_FREE = B_S_FULL + NS, B_P_FULL = B_S_FREE + NS, B_O_FREE = B_P_FULL + NS,
                         B_ITEM_FULL = B_O_FREE + 1, B_ITEM_EMPTY = B_ITEM_FULL + 2, B_PAIR = B_ITEM_EMPTY + 2,
                         B_HAND = B_PAIR + 4, B_EPI = B_HAND + 8, B_DRAIN = B_EPI + 1, N_BARS = B_DRAIN + 2;
    static constexpr uint32_t item_off = bar_off + ((N_BARS * 8 + 15) / 16) * 16;
    static constexpr uint32_t hand_off = item_off + 2 * sizeof(ItemInfo);   // float [4 quadrants][2 slots][32]
    static constexpr uint32_t xchg_off = hand_off + 4 * 2 * 32 * sizeof(float);   // float [2 warps][128 rows]
    static constexpr uint32_t misc_off = xchg_off + 2 * kRows * sizeof(float);
    static constexpr uint32_t bytes = misc_off + 16;         // tmem holder, abort flag
    // The dynamic shared-memory window starts 1024-byte aligned (no static
    // shared memory precedes it); the kernel checks this and aborts if not.
    static constexpr uint32_t smem_request = bytes;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 384;                   // S buffer s at column 128 * s
};

constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = 8;    // warp w: TMEM lanes 32 * (w % 4), S columns 64 * (w / 4)
constexpr int kProducerWarp = 8;
constexpr int kQkWarp = 9;
constexpr int kPvWarp = 10;
constexpr int kVProducerWarp = 11;
constexpr int kLaunchRegs = 168;            // per thread at launch: 384 x 168 = 64512
constexpr uint32_t kSoftmaxRegs = 216;      // warpgroups 0-1 after setmaxnreg
constexpr uint32_t kOtherRegs = 72;         // warpgroup 2 (producers, issuers)
static_assert(256 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs, "register split");
constexpr float kNegInf = -__builtin_huge_valf();

// Wait that ignores the abort flag: used only to drain in-flight copies.
__device__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kDrainTimeoutNs) return false;
    return true;
}

// Block-table entries of a few consecutive prefix tiles of one sequence,
// one page a lane: lane j holds page (t0 << (7 - page_lg)) + j, clamped to
// the sequence's last page, so no entry past the prefix is read. One load
// serves 32 pages (4 tiles of 16-row pages), and a producer issues it before
// its wait on the ring stage so that the read overlaps the wait.
struct PageWindow {
    int b = -1, t0 = 0, phys = 0;
    // Make tile t of sequence b (prefix length P) covered; whole warp.
    __device__ __forceinline__ void cover(const AttnArgs &a, int b_, int P, int t, int lane) {
        const int lg = a.page_lg, span = 32 >> (7 - lg);
        if (b_ == b && t >= t0 && t < t0 + span) return;
        const int last = max(0, ((P + (1 << lg) - 1) >> lg) - 1);
        b = b_;
        t0 = t;
        phys = a.block_table[(size_t)b_ * a.pages_per_seq + min((t << (7 - lg)) + lane, last)];
    }
    // The physical page that lane loads for tile t (covered); whole warp.
    __device__ __forceinline__ int page_of(const AttnArgs &a, int t, int lane) const {
        return __shfl_sync(0xffffffffu, phys, (((t - t0) << (7 - a.page_lg)) + lane) & 31);
    }
};

// Prefix tile t of KV head kh of sequence b (keys t * 128 ..) into the
// shared tile at dst: one box per 64 columns from the contiguous cache, or,
// paged, one box per page and 64 columns, lane j loading page j, whose
// physical number `phys` the caller took from its PageWindow. Pages past
// the sequence's last one (the tile's ragged end, masked later) reload that
// last page. Called by the whole warp after lane 0 has set the barrier's
// expected bytes.
template <int D, bool kPaged>
__device__ __forceinline__ void load_prefix_tile(const CUtensorMap *map, const AttnArgs &a, const Layout &L,
                                                 uint32_t dst, int b, int kh, int t, int phys, uint32_t bar,
                                                 int lane) {
    using C = AttnCfg<D>;
    if (!kPaged) {
        if (lane == 0)
            for (int dc = 0; dc < C::kBoxes; ++dc)
                tma_load_3d(dst + dc * (kBN * 128), map, dc * 64, t * kBN, b * L.Hkv + kh, bar);
        return;
    }
    const int lg = a.page_lg, per_tile = kBN >> lg;
    if (lane < per_tile) {
        for (int dc = 0; dc < C::kBoxes; ++dc)
            tma_load_3d(dst + dc * (kBN * 128) + (lane << lg) * 128, map, dc * 64, kh, phys << lg, bar);
    }
}

template <int D, bool kPaged>
__device__ __forceinline__ void producer_loop(const AttnMaps &maps, const Layout &L, const AttnArgs &a,
                                              uint32_t sbase, uint32_t bars, ItemInfo *items_s,
                                              volatile int *abort) {
    using C = AttnCfg<D>;
    const int lane = threadIdx.x & 31;
    QTile *qtab = reinterpret_cast<QTile *>(a.ws + L.qtab_off);
    auto bar = [&](int i) { return bars + 8u * i; };
    // This CTA's stream-K range of the concatenated unit tiles, derived here
    // from prefix_lens and n_nodes (no earlier kernel needed).
    const int c = blockIdx.x;
    const PlanSeq ps = plan_locate(L, a.prefix_lens, a.n_nodes, c, a.num_ctas);
    const int alpha = ps.alpha;
    const int hi = ps.hi;
    int lo = ps.lo;
    // The unit (b, kh, qt) holding virtual tile lo, and its first virtual
    // tile S (its real tiles start at S + alpha).
    int b = ps.b, kh = 0, qt = 0, P = ps.P, n = ps.n;
    int S = 0;
    if (lo < hi) {
        if (b < 0) {
            lo = hi;                        // unreachable for a consistent plan
        } else {
            const int th = head_tiles(P, n, L) + alpha * head_units(n, L);
            kh = (lo - ps.seq_start) / th;
            S = ps.seq_start + kh * th;
            for (int us = unit_tiles(P, n, 0, L) + alpha; S + us <= lo && qt + 1 < L.QT;
                 us = unit_tiles(P, n, qt, L) + alpha) {
                S += us;
                ++qt;
            }
        }
    }
    int ic = 0, qc = 0, kc = 0;
    bool ok = true;
    // K tile t of the current item into the next ring stage.
    int skipped = -1;                   // a load left out on purpose (stall-test build only)
    PageWindow pw;
    auto issue_k = [&](const ItemInfo &info, int t) -> bool {
        const bool tree = t >= info.t_pre;
        const bool paged = kPaged && !tree;
        const int ks = kc % C::NK;
        const int pt = tree ? 0 : prefix_tile(info, t);
        if (paged) pw.cover(a, info.b, info.P, pt, lane);
        if (!mbar_wait(bar(C::B_K_EMPTY + ks), ((kc / C::NK) & 1) ^ 1, abort, a.status)) return false;
#ifdef JF_STALL_TEST
        if (kc == 0) {                  // never arrives: the first QK^T waits until its limit
            skipped = 0;
            ++kc;
            return true;
        }
#endif
        if (lane == 0) mbar_arrive_expect_tx(bar(C::B_K_FULL + ks), C::kTileBytes);
        __syncwarp();
        const uint32_t dst = sbase + C::k_off + ks * C::kTileBytes;
        if (tree) {
            if (lane == 0)
                for (int dc = 0; dc < C::kBoxes; ++dc)
                    tma_load_3d(dst + dc * (kBN * 128), &maps.tree_k, dc * 64, info.kh,
                                info.b * L.Nmax + (t - info.t_pre) * kBN, bar(C::B_K_FULL + ks));
        } else {
            load_prefix_tile<D, kPaged>(&maps.k_cache, a, L, dst, info.b, info.kh, pt,
                                        paged ? pw.page_of(a, pt, lane) : 0,
                                        bar(C::B_K_FULL + ks), lane);
        }
        __syncwarp();
        ++kc;
        return true;
    };
    while (ok) {
        const int slot = ic & 1;
        if (!mbar_wait(bar(C::B_ITEM_EMPTY + slot), ((ic >> 1) & 1) ^ 1, abort, a.status)) break;
        ItemInfo info{};
        int t_next = 0;
        if (lo < hi) {                      // skip the unit's virtual tiles
            if (S + alpha >= hi) lo = hi;
            else if (lo < S + alpha) lo = S + alpha;
        }
        if (lo < hi) {
            const int T = unit_tiles(P, n, qt, L);
            S += alpha;                     // S: the unit's first real tile
            const int u = (b * L.Hkv + kh) * L.QT + qt;
            info.valid = 1;
            info.qtile = u;
            info.b = b;
            info.kh = kh;
            info.qt = qt;
            info.tb = lo - S;
            info.te = min(hi, S + T) - S;
            info.P = P;
            info.n = n;
            info.t_pre = ceil_div(P, kBN);
            // The first range boundary inside the unit's prefix tiles, if
            // any, falls on prefix tile 0 (see prefix_tile): the first CTA
            // whose range starts after S is the smallest c with
            // c * total >= (S + 1) * C.
            info.rot = 0;
            if (info.t_pre > 1 && (long long)ps.kv_tiles * 2 * C::kTileBytes > kRotateBytes) {
                const long long total = (long long)ps.n_ctas * ps.qt + ps.rt;
                const int c1 = (int)(((long long)(S + 1) * ps.n_ctas + total - 1) / total);
                if (c1 < ps.n_ctas) {
                    const int s1 = range_start(c1, ps.qt, ps.rt, ps.n_ctas) - S;
                    if (s1 < info.t_pre) info.rot = info.t_pre - s1;
                }
            }
            // Q and the first K tiles go out before the rest of the item's
            // bookkeeping, so that their latency overlaps it.
            const int qb = qc % C::NQ;
            if (!mbar_wait(bar(C::B_Q_EMPTY + qb), ((qc / C::NQ) & 1) ^ 1, abort, a.status)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(C::B_Q_FULL + qb), C::kQBytes);
                for (int dc = 0; dc < C::kBoxes; ++dc)
                    tma_load_3d(sbase + C::q_off + qb * C::kQBytes + dc * C::kQBoxBytes, &maps.q, dc * 64,
                                info.kh * L.G, info.b * L.Nmax + info.qt * L.NB, bar(C::B_Q_FULL + qb));
            }
            ++qc;
            t_next = info.tb;
            for (; t_next < info.te && t_next < info.tb + C::NK && ok; ++t_next) ok = issue_k(info, t_next);
            if (!ok) break;
            const int c_first = cta_of_tile(S, ps.qt, ps.rt, ps.n_ctas);
            info.ns = cta_of_tile(S + T - 1, ps.qt, ps.rt, ps.n_ctas) - c_first + 1;
            // A split unit is at most this CTA's first item (slot 2c) or its
            // last (slot 2c + 1): units in between lie wholly in the range.
            info.slot = info.ns > 1 ? 2 * c + (ic > 0 ? 1 : 0) : -1;
            if (info.tb == 0 && lane == 0)  // the unit starts in this range: record its split plan
                qtab[u] = QTile{info.ns, c, ic == 0 ? 1 : 0, S};
            lo = S + info.te;
            S += T;
            if (lo < hi) {                  // the next unit with tiles
                if ((qt + 1) * L.NB < n) {
                    ++qt;
                } else {
                    qt = 0;
                    if (kh + 1 < L.Hkv) {
                        ++kh;
                    } else {
                        kh = 0;
                        for (++b; b < L.B; ++b) {
                            P = a.prefix_lens[b];
                            n = a.n_nodes[b];
                            if (seq_valid(P, n, L)) break;
                        }
                        if (b >= L.B) lo = hi;  // unreachable for a consistent plan
                    }
                }
            }
        }
        if (lane == 0) {
            items_s[slot] = info;
            mbar_arrive(bar(C::B_ITEM_FULL + slot));
        }
        __syncwarp();
        ++ic;
        if (!info.valid) break;
        for (; t_next < info.te; ++t_next)
            if (!issue_k(info, t_next)) { ok = false; break; }
    }
    if (*abort && lane == 0) {
        // Let every copy this warp started land before the CTA can exit.
        for (int s = 0; s < C::NQ; ++s)
            if (qc > s) mbar_wait_drain(bar(C::B_Q_FULL + s), (((qc - 1 - s) / C::NQ)) & 1);
        for (int s = 0; s < C::NK; ++s) {
            const int k = (kc - 1) - ((kc - 1 - s) % C::NK + C::NK) % C::NK;   // last load into stage (k % NK == s)
            if (kc > s && k != skipped) mbar_wait_drain(bar(C::B_K_FULL + s), (k / C::NK) & 1);
        }
    }
}

// Item hand-off shared by the two issuers: returns false at the end.
template <int D>
__device__ __forceinline__ bool next_item(uint32_t bars, const ItemInfo *items_s, int &ic, ItemInfo &info,
                                          volatile int *abort, int32_t *status) {
    using C = AttnCfg<D>;
    const int slot = ic & 1;
    if (!mbar_wait(bars + 8u * (C::B_ITEM_FULL + slot), (ic >> 1) & 1, abort, status)) return false;
    info = items_s[slot];
    ++ic;
    return info.valid != 0;
}

// V producer: the V tiles of each item into the NV-stage ring. It runs apart
// from the Q/K producer so that a K load never waits behind a V stage that a
// slower PV still holds.
template <int D, bool kPaged>
__device__ __forceinline__ void v_producer_loop(const AttnMaps &maps, const Layout &L, const AttnArgs &a,
                                                uint32_t sbase, uint32_t bars, const ItemInfo *items_s,
                                                volatile int *abort) {
    using C = AttnCfg<D>;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return bars + 8u * i; };
    int ic = 0, vc = 0;
    ItemInfo info;
    bool ok = true;
    PageWindow pw;
    while (ok && next_item<D>(bars, items_s, ic, info, abort, a.status)) {
        const int slot = (ic - 1) & 1;
        {
            for (int t = info.tb; t < info.te; ++t) {
                const bool tree = t >= info.t_pre;
                const bool paged = kPaged && !tree;
                const int vs = vc % C::NV;
                const int pt = tree ? 0 : prefix_tile(info, t);
                if (paged) pw.cover(a, info.b, info.P, pt, lane);
                if (!mbar_wait(bar(C::B_V_EMPTY + vs), ((vc / C::NV) & 1) ^ 1, abort, a.status)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(bar(C::B_V_FULL + vs), C::kTileBytes);
                __syncwarp();
                const uint32_t dst = sbase + C::v_off + vs * C::kTileBytes;
                if (tree) {
                    if (lane == 0)
                        for (int dc = 0; dc < C::kBoxes; ++dc)
                            tma_load_3d(dst + dc * (kBN * 128), &maps.tree_v, dc * 64, info.kh,
                                        info.b * L.Nmax + (t - info.t_pre) * kBN, bar(C::B_V_FULL + vs));
                } else {
                    load_prefix_tile<D, kPaged>(&maps.v_cache, a, L, dst, info.b, info.kh, pt,
                                        paged ? pw.page_of(a, pt, lane) : 0, bar(C::B_V_FULL + vs), lane);
                }
                __syncwarp();
                ++vc;
            }
        }
        if (ok && lane == 0) mbar_arrive(bar(C::B_ITEM_EMPTY + slot));
    }
    if (*abort && lane == 0) {
        // Let every copy this warp started land before the CTA can exit.
        for (int s = 0; s < C::NV; ++s)
            if (vc > s) mbar_wait_drain(bar(C::B_V_FULL + s), (((vc - 1 - s) / C::NV)) & 1);
    }
}

// QK^T issuer: S(g) = Q K(g)^T into S buffer g % 3, up to 2 tiles ahead.
template <int D>
__device__ __forceinline__ void qk_loop(const AttnArgs &a, uint32_t sbase, uint32_t bars, const ItemInfo *items_s,
                                        uint32_t tmem, volatile int *abort) {
    using C = AttnCfg<D>;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return bars + 8u * i; };
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
    // Descriptors are built once; the start-address field (address >> 4, in
    // the low bits) is then advanced by adding byte offsets >> 4.
    const uint64_t q_desc = sdesc_sw128(sbase + C::q_off, 16, 1024);
    const uint64_t k_desc = sdesc_sw128(sbase + C::k_off, 16, 1024);
    int ic = 0, qc = 0, kc = 0, g = 0;
    ItemInfo info;
    bool ok = true;
    while (ok && next_item<D>(bars, items_s, ic, info, abort, a.status)) {
        const int slot = (ic - 1) & 1;
        const int qb = qc % C::NQ;
        if (!mbar_wait(bar(C::B_Q_FULL + qb), (qc / C::NQ) & 1, abort, a.status)) break;
        ++qc;
        const uint64_t qd = q_desc + ((qb * C::kQBytes) >> 4);
        const int nt = info.te - info.tb;
        for (int j = 0; j < nt; ++j, ++kc, ++g) {
            const int ks = kc % C::NK, sb = g % C::NS;
            if (!mbar_wait(bar(C::B_K_FULL + ks), (kc / C::NK) & 1, abort, a.status) ||
                !mbar_wait(bar(C::B_S_FREE + sb), ((g / C::NS) & 1) ^ 1, abort, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            __syncwarp();
            const uint64_t b0 = k_desc + ((ks * C::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + sb * 128, qd + (((kk >> 2) * C::kQBoxBytes + (kk & 3) * 32) >> 4),
                       b0 + (((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
            mma_commit(bar(C::B_S_FULL + sb));
            mma_commit(bar(C::B_K_EMPTY + ks));
        }
        if (ok && lane == 0) mbar_arrive(bar(C::B_ITEM_EMPTY + slot));
    }
    // Every MMA this warp issued has completed before the CTA can free TMEM
    // or exit, on every path (an abort included).
    mma_commit(bar(C::B_DRAIN + 0));
    if (lane == 0) mbar_wait_drain(bar(C::B_DRAIN + 0), 0);
    __syncwarp();
}

// PV issuer: O (+)= P(g) V(g); a buffer's S/P slot returns to the QK issuer
// when this PV completes.
template <int D>
__device__ __forceinline__ void pv_loop(const AttnArgs &a, uint8_t *smem, uint32_t sbase, uint32_t bars,
                                        const ItemInfo *items_s, uint32_t tmem, volatile int *abort) {
    using C = AttnCfg<D>;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return bars + 8u * i; };
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, false, true);
    const uint64_t v_desc = sdesc_sw128(sbase + C::v_off, kBN * 128, 1024);
    int ic = 0, vc = 0, g = 0, items = 0;
    ItemInfo info;
    bool ok = true;
    while (ok && next_item<D>(bars, items_s, ic, info, abort, a.status)) {
        const int slot = (ic - 1) & 1;
        // The first PV of an item overwrites O: every softmax warp must have
        // read the previous item's O first.
        if (items > 0 && !mbar_wait(bar(C::B_O_FREE), (items - 1) & 1, abort, a.status)) break;
        ++items;
        const int nt = info.te - info.tb;
        for (int j = 0; j < nt; ++j, ++vc, ++g) {
            const int vs = vc % C::NV, sb = g % C::NS;
            // V has long landed when P is ready: wait for it first, so that
            // the PV goes out the moment the softmax hands P over.
            if (!mbar_wait(bar(C::B_V_FULL + vs), (vc / C::NV) & 1, abort, a.status) ||
                !mbar_wait(bar(C::B_P_FULL + sb), (g / C::NS) & 1, abort, a.status)) {
                ok = false;
                break;
            }
            // V rows past the prefix length / past n_nodes: zero them so that
            // whatever the caller's memory holds there cannot reach O via 0 * NaN.
            const int t = info.tb + j;
            int r0 = kBN;
            if (t < info.t_pre) {
                if (prefix_tile(info, t) == info.t_pre - 1 && (info.P % kBN) != 0) r0 = info.P % kBN;
            } else {
                const int left = info.n - (t - info.t_pre) * kBN;
                r0 = left < 0 ? 0 : (left < kBN ? left : kBN);
            }
            if (r0 < kBN) {
                const int chunks = (kBN - r0) * 8;            // 16-byte chunks per box
                for (int dc = 0; dc < C::kBoxes; ++dc) {
                    uint4 *base = reinterpret_cast<uint4 *>(smem + C::v_off + vs * C::kTileBytes + dc * (kBN * 128) +
                                                            r0 * 128);
                    for (int c = lane; c < chunks; c += 32) base[c] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            __syncwarp();
            const uint64_t b0 = v_desc + ((vs * C::kTileBytes) >> 4);
            // P of keys 16kk..16kk+15: bf16 pairs at S columns 8kk..8kk+7
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts(tmem + C::kColO, tmem + sb * 128 + kk * 8, b0 + ((kk * 2048) >> 4), idesc_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar(C::B_S_FREE + sb));
            mma_commit(bar(C::B_V_EMPTY + vs));
        }
        if (ok && lane == 0) mbar_arrive(bar(C::B_ITEM_EMPTY + slot));
    }
    // Every MMA this warp issued has completed before the CTA can free TMEM
    // or exit, on every path (an abort included).
    mma_commit(bar(C::B_DRAIN + 1));
    if (lane == 0) mbar_wait_drain(bar(C::B_DRAIN + 1), 0);
    __syncwarp();
}

// Ancestor mask ("JetFlow: Scaling Speculative Decoding with Parallel Tree
// Drafting", blog, section "What JetFlow Does Differently": a node attends to
// its ancestors, never to siblings or descendants). Bit k of the result is
// set iff tree key k0 + k (k < 128) is the node itself or one of its
// ancestors. The walk follows parents from the node toward the root and
// stops below k0; indices strictly decrease along it, so it ends after at
// most kMaxNodes steps even on a malformed tree (whose output the combine
// kernel then replaces with NaN).
__device__ __forceinline__ uint4 ancestor_bits(const int32_t *parents, int node, int k0) {
    uint32_t w0 = 0u, w1 = 0u, w2 = 0u, w3 = 0u;
    int j = node;
    for (int hop = 0; hop < kMaxNodes && j >= k0; ++hop) {
        const int k = j - k0;
        if (k < kBN) {
            const uint32_t bit = 1u << (k & 31);
            w0 |= (k >> 5) == 0 ? bit : 0u;
            w1 |= (k >> 5) == 1 ? bit : 0u;
            w2 |= (k >> 5) == 2 ? bit : 0u;
            w3 |= (k >> 5) == 3 ? bit : 0u;
        }
        const int p = __ldg(parents + j);
        j = p < j ? p : -1;
    }
    return make_uint4(w0, w1, w2, w3);
}

// Softmax and epilogue. The two warps of a row quadrant (q and q + 4, both
// on TMEM lanes 32q..32q+31) take alternate key tiles: warp q + 4p owns the
// tiles of global index g with g % 2 == p and does the whole 128-column row
// of its tiles. One warp's TMEM-load and reduction latency then overlaps the
// other's ex2 work, instead of both warps running the same phase together.
//
// The running max is the one piece of state that crosses tiles. The owner of
// tile g publishes m(g) to its partner right after its row max (hand-off slot
// g % 2 of the quadrant, a bounded mbarrier); the owner of tile g + 1 reads it
// before its exps. Each warp keeps its own part of the row sum, l_own, with
// the reference max it is expressed in; the two parts are merged in the
// epilogue. O is rescaled, when needed, by the owner of the tile that raised
// the max, after the PV of the previous tile has completed.
//
// The warp reads the tile's whole 128-key row once for the row max, then
// runs the exp pass over 64-column chunks read again from TMEM. The softmax
// warpgroups get 216 registers per thread (setmaxnreg), the producer and
// issuer warpgroup 72. P (bf16 pairs) goes back over the S columns 0-63 of
// its buffer.
template <int D>
__device__ __forceinline__ void softmax_loop(const AttnMaps &maps, const Layout &L, const AttnArgs &a,
                                             uint8_t *smem, uint32_t bars, const ItemInfo *items_s, float *hand,
                                             float *xchg, uint32_t tmem, volatile int *abort) {
    using C = AttnCfg<D>;
    constexpr int kOHalf = D / 2;                   // O columns per warp in the epilogue
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, par = warp >> 2;        // row quadrant, tile parity (= epilogue column half)
    const int r = q * 32 + lane;                    // stacked row = TMEM lane
    auto bar = [&](int i) { return bars + 8u * i; };
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t t_o = t_row + C::kColO;
    __half *opart = reinterpret_cast<__half *>(a.ws + L.opart_off);
    float *mlpart = reinterpret_cast<float *>(a.ws + L.ml_off);   // (m, l, e0, e1) per piece row
    float *hand_q = hand + q * 64;
    const float sl2 = a.scale_log2;
    int ic = 0, g = 0, xc = 0, items = 0;
    int pending_q = -1;         // thread 0: Q buffer whose TMA store has not yet read it back

    // Thread 0 hands a staging buffer back to the producer once the bulk
    // store that reads it has done so.
    auto release_q = [&]() {
        if (threadIdx.x == 0 && pending_q >= 0) {
            bulk_wait_read();
            mbar_arrive(bar(C::B_Q_EMPTY + pending_q));
            pending_q = -1;
        }
    };
    auto publish = [&](int gg, float m) {
        hand_q[(gg & 1) * 32 + lane] = m;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_HAND + q * 2 + (gg & 1)));
    };
    auto receive = [&](int gg, float &m) -> bool {
        if (!mbar_wait(bar(C::B_HAND + q * 2 + (gg & 1)), (gg >> 1) & 1, abort, a.status)) return false;
        m = hand_q[(gg & 1) * 32 + lane];
        return true;
    };
    // PV of tile gg has completed (its S buffer was handed back).
    auto wait_pv = [&](int gg) {
        return mbar_wait(bar(C::B_S_FREE + gg % C::NS), (gg / C::NS) & 1, abort, a.status);
    };
    // -inf on keys this row may not see: not an ancestor (tree tile, one mask
    // bit per key) or past the prefix length (lim keys valid).
    auto mask128 = [&](uint32_t (&sv)[kBN], bool tree, const uint4 &mw, int lim) {
        if (tree) {
            const uint32_t w[4] = {mw.x, mw.y, mw.z, mw.w};
#pragma unroll
            for (int c = 0; c < kBN; ++c)
                if (!((w[c >> 5] >> (c & 31)) & 1u)) sv[c] = __float_as_uint(kNegInf);
        } else if (lim < kBN) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
                if (c >= lim) sv[c] = __float_as_uint(kNegInf);
        }
    };
    auto max128 = [&](const uint32_t (&sv)[kBN]) {
        float m4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = __uint_as_float(sv[k]);
#pragma unroll
        for (int c = 4; c < kBN - 4; c += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                m4[k] = max3f(m4[k], __uint_as_float(sv[c + k]), __uint_as_float(sv[c + 4 + k]));
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmaxf(m4[k], __uint_as_float(sv[kBN - 4 + k]));
        return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    };
    while (true) {
        const int slot = ic & 1;
        if (!mbar_wait(bar(C::B_ITEM_FULL + slot), (ic >> 1) & 1, abort, a.status)) break;
        const ItemInfo info = items_s[slot];
        ++ic;
        if (!info.valid) break;
        const int node = (info.qt << L.lgNB) + (r >> L.lgG);
        const int head = (info.kh << L.lgG) + (r & (L.G - 1));
        const bool row_valid = node < info.n;
        const int32_t *par_b = a.parents + (size_t)info.b * L.Nmax;
        // The ancestor walks of the item's tree tiles read this sequence's
        // parents (at most 1 KB): start pulling them into L1 now.
        if (info.te > info.t_pre && lane < ceil_div(L.Nmax, 32)) prefetch_l1(par_b + 32 * lane);
        float m_run = kNegInf;                      // reference of O after this warp's last tile
        float m_own = kNegInf, l_own = 0.f;         // this warp's part of the row sum, and its reference
        const int nt = info.te - info.tb;
        bool fail = false;
        for (int j = 0; j < nt; ++j, ++g) {
            if ((g & 1) != par) continue;                  // the partner's tile
            const int t = info.tb + j;
            const bool tree = t >= info.t_pre;
            uint4 mw = make_uint4(0u, 0u, 0u, 0u);         // ancestor bits of the tile's 128 keys
            if (tree && row_valid) mw = ancestor_bits(par_b, node, (t - info.t_pre) * kBN);
            const int lim = (!tree && prefix_tile(info, t) == info.t_pre - 1) ? info.P - (info.t_pre - 1) * kBN : kBN;
            const int sb = g % C::NS;
            const uint32_t t_s = t_row + sb * 128;
            // The running max so far, published by the previous tile's owner
            // long before this tile's S is ready: taken before waiting for S,
            // so that it is off the tile's critical path.
            float m_prev = kNegInf;
            if (j > 0 && !receive(g - 1, m_prev)) { fail = true; break; }
            if (!mbar_wait(bar(C::B_S_FULL + sb), (g / C::NS) & 1, abort, a.status)) { fail = true; break; }
            tc_fence_after();
            float mt;
            {
                uint32_t sv[kBN];                          // the whole row of the tile
                tmem_ld128(t_s, sv);
                if (tree || lim < kBN) {                   // rare: write the masked row back for the exp pass
                    mask128(sv, tree, mw, lim);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) tmem_st32(t_s + 32 * c4, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c4]));
                    tmem_wait_st();
                }
                mt = max128(sv) * sl2;
            }
            float m_new = mt;
            bool need = false;
            if (j > 0) {
                m_new = fmaxf(m_prev, mt);
                need = m_new > m_prev + 8.0f;              // lazy: O keeps m_prev unless it grows > 2^8
                if (!need) m_new = m_prev;
            }
            publish(g, m_new);                             // the partner's next tile can go on
            if (j > 0) {
                if (__any_sync(0xffffffffu, need)) {
                    // O holds PV up to the previous tile: wait for it, then
                    // rescale the quadrant's rows in place.
                    if (!wait_pv(g - 1)) { fail = true; break; }
                    tc_fence_after();
                    const float alpha = need ? ex2_approx(m_prev - m_new) : 1.0f;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(t_o + c * 32, v);
#pragma unroll
                        for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                        tmem_st32(t_o + c * 32, v);
                    }
                }
            }
            m_run = m_new;
            if (m_own != m_run) {                          // bring l_own to the new reference
                l_own *= ex2_approx(m_own - m_run);        // l_own = 0 while m_own = -inf
                m_own = m_run;
            }
            const float neg_m = (m_run == kNegInf) ? 0.f : -m_run;
            // exp pass in two rolled 64-key chunks, each read again from
            // TMEM: one copy of the exp code keeps the hot loop small. The
            // scaling and the sums use packed f32x2 arithmetic (one
            // instruction per key pair).
            const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(neg_m, neg_m);
            uint64_t lsum2 = f32x2(0.f, 0.f);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t sh[64];
                tmem_ld64(t_s + 64 * h, sh);
                uint32_t pv[32];
                uint64_t sum2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float2 x = unpack_f32x2(fma_f32x2(f32x2(sh[c], sh[c + 1]), sl2x2, negm2));
                    const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                    sum2[(c >> 1) & 1] = add_f32x2(sum2[(c >> 1) & 1], f32x2(p0, p1));
                    pv[c >> 1] = pack_bf16x2(p0, p1);
                }
                lsum2 = add_f32x2(lsum2, add_f32x2(sum2[0], sum2[1]));
                tmem_st32(t_s + 32 * h, pv);               // P of keys 64h.. -> S columns 32h..
            }
            const float2 ls = unpack_f32x2(lsum2);
            l_own += ls.x + ls.y;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_P_FULL + sb));
            release_q();                                   // a staged output store has long read its buffer
        }
        if (fail) break;
        // Epilogue. The final max is m(g_last), published by the last tile's
        // owner; the partner is the reader its hand-off slot expects.
        release_q();
        const int g_last = g - 1;
        float m_fin = m_run;
        if ((g_last & 1) != par && !receive(g_last, m_fin)) break;
        const float l_mine = (m_own == m_fin) ? l_own : l_own * ex2_approx(m_own - m_fin);
        // The last PV of the item has completed: O is final, and the partner
        // cannot reach its next epilogue (which would reuse xchg) before this
        // warp has read xchg and released O.
        if (!wait_pv(g_last)) break;
        tc_fence_after();
        xchg[par * kRows + r] = l_mine;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PAIR + q));
        if (!mbar_wait(bar(C::B_PAIR + q), xc & 1, abort, a.status)) break;
        ++xc;
        const float l_run = l_mine + xchg[(par ^ 1) * kRows + r];
        // This warp's half of the row; then O's TMEM belongs to the next item.
        uint32_t ov[kOHalf];
        if constexpr (kOHalf == 64)
            tmem_ld64(t_o + par * kOHalf, ov);
        else
            tmem_ld32(t_o + par * kOHalf, ov);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_O_FREE));
        // Final rows are bf16. The pieces of a split unit are fp16 rows divided
        // by their own l and scaled by 2^-e, e chosen per half row (this
        // warp's columns) so that the largest magnitude lies in [2^14, 2^15):
        // fp16's range then holds any bf16 value, and the merge multiplies by
        // 2^e again. (m, l, e0, e1) go beside them.
        const bool split = info.ns > 1;
        const float inv_l = 1.0f / l_run;
        int e_half = 0;
        // Scaled and packed in place: ov[2k] holds the pair for columns 2k, 2k+1.
        if (split) {
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < kOHalf; ++k) amax = fmaxf(amax, fabsf(__uint_as_float(ov[k])));
            amax *= inv_l;
            if (amax > 0.f && amax <= 3.4e38f)
                e_half = min(max(((__float_as_int(amax) >> 23) & 0xFF) - 127 - 14, -100), 100);
            const float sc = inv_l * __int_as_float((127 - e_half) << 23);    // inv_l * 2^-e, exact
#pragma unroll
            for (int e = 0; e < kOHalf / 2; ++e) {
                const __half2 h = __floats2half2_rn(__uint_as_float(ov[2 * e]) * sc, __uint_as_float(ov[2 * e + 1]) * sc);
                ov[e] = *reinterpret_cast<const uint32_t *>(&h);
            }
        } else {
#pragma unroll
            for (int e = 0; e < kOHalf / 2; ++e)
                ov[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
        }
        auto pack8 = [&](int k) { return make_uint4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]); };
        // A unit whose rows are all real nodes is staged in its own Q buffer
        // (free since its last QK^T) in the 128-byte-swizzled box layout and
        // written by TMA bulk stores: one wide store instead of 32 scattered
        // rows per warp instruction. Other units write their valid rows
        // directly.
        const bool whole = (info.qt + 1) * L.NB <= info.n;
        const int qb = items % C::NQ;
        if (whole) {
            uint8_t *row = smem + C::q_off + qb * C::kQBytes + ((par * kOHalf) / 64) * C::kQBoxBytes + r * 128;
            const int c0 = ((par * kOHalf) % 64) / 8;      // first 16-byte chunk of this warp's columns
#pragma unroll
            for (int k = 0; k < kOHalf / 8; ++k)
                *reinterpret_cast<uint4 *>(row + (((c0 + k) ^ (r & 7)) << 4)) = pack8(k);
            fence_proxy_async_smem();
        } else if (row_valid) {
            uint4 *dst = split ? reinterpret_cast<uint4 *>(opart + ((size_t)info.slot * kRows + r) * D + par * kOHalf)
                               : reinterpret_cast<uint4 *>(a.out + (((size_t)info.b * L.Nmax + node) * L.Hq + head) * D +
                                                           par * kOHalf);
#pragma unroll
            for (int k = 0; k < kOHalf / 8; ++k) dst[k] = pack8(k);
        }
        if (split) {
            float *rec = mlpart + 4 * ((size_t)info.slot * kRows + r);
            if (par == 0) {
                rec[0] = m_fin;
                rec[1] = l_run;
            }
            rec[2 + par] = (float)e_half;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_EPI));
        bool ok_epi = true;
        if (threadIdx.x == 0) {
            ok_epi = mbar_wait(bar(C::B_EPI), items & 1, abort, a.status);
            if (ok_epi && whole) {
                const uint32_t src = smem_u32(smem + C::q_off + qb * C::kQBytes);
                for (int dc = 0; dc < C::kBoxes; ++dc) {
                    if (split)
                        tma_store_3d(&maps.part, src + dc * C::kQBoxBytes, dc * 64, 0, info.slot);
                    else
                        tma_store_3d(&maps.out, src + dc * C::kQBoxBytes, dc * 64, info.kh * L.G,
                                     info.b * L.Nmax + info.qt * L.NB);
                }
                bulk_commit();
                pending_q = qb;
            } else if (ok_epi) {
                mbar_arrive(bar(C::B_Q_EMPTY + qb));
            }
        }
        if (warp == 0) ok_epi = __shfl_sync(0xffffffffu, ok_epi ? 1 : 0, 0) != 0;
        if (!ok_epi) break;
        ++items;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_ITEM_EMPTY + slot));
    }
    // Every bulk store of this CTA has landed before it can exit.
    if (threadIdx.x == 0) {
        if (pending_q >= 0) {
            bulk_wait_read();
            mbar_arrive(bar(C::B_Q_EMPTY + pending_q));
        }
        bulk_wait_all();
    }
}

template <int D, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    tree_attention_kernel(const __grid_constant__ AttnMaps maps, const Layout L, const AttnArgs a) {
    using C = AttnCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const int warp = threadIdx.x >> 5;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + C::bar_off;
    ItemInfo *items_s = reinterpret_cast<ItemInfo *>(smem + C::item_off);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::misc_off + 4);

    if (smem_u32(smem) & 1023u) {   // swizzled TMA tiles need 1024-byte alignment
        if (threadIdx.x == 0) set_status(a.status, JF_STATUS_TIMEOUT);
        return;
    }
    if (threadIdx.x == 0) {
        auto init = [&](int i, uint32_t count) { mbar_init(bars + 8u * i, count); };
        for (int s = 0; s < C::NQ; ++s) { init(C::B_Q_FULL + s, 1); init(C::B_Q_EMPTY + s, 1); }
        for (int s = 0; s < C::NK; ++s) { init(C::B_K_FULL + s, 1); init(C::B_K_EMPTY + s, 1); }
        for (int s = 0; s < C::NV; ++s) { init(C::B_V_FULL + s, 1); init(C::B_V_EMPTY + s, 1); }
        for (int s = 0; s < C::NS; ++s) {
            init(C::B_S_FULL + s, 1);
            init(C::B_S_FREE + s, 1);
            init(C::B_P_FULL + s, kSoftmaxWarps / 2);      // the tile's owner in each row quadrant
        }
        init(C::B_O_FREE, kSoftmaxWarps);
        for (int s = 0; s < 2; ++s) {
            init(C::B_ITEM_FULL + s, 1);
            init(C::B_ITEM_EMPTY + s, 3 + kSoftmaxWarps);  // both issuers, the V producer, every softmax warp
        }
        for (int q = 0; q < 4; ++q) init(C::B_PAIR + q, 2); // the two warps that share a row quadrant
        for (int h = 0; h < 8; ++h) init(C::B_HAND + h, 1); // row-max hand-off, [quadrant][tile parity]
        init(C::B_EPI, kSoftmaxWarps);                     // an item's output is staged
        init(C::B_DRAIN + 0, 1);                           // the QK^T issuer's MMAs have completed
        init(C::B_DRAIN + 1, 1);                           // the PV issuer's MMAs have completed
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp) {
        // The plan's first loads after the wait: start them towards L2 now.
        const int lane = threadIdx.x & 31;
        if (32 * lane < L.B) {
            prefetch_l2(a.prefix_lens + 32 * lane);
            prefetch_l2(a.n_nodes + 32 * lane);
        }
    }
    if (warp == kProducerWarp && (threadIdx.x & 31) == 0) {
        tma_prefetch_map(&maps.q);
        tma_prefetch_map(&maps.k_cache);
        tma_prefetch_map(&maps.v_cache);
        tma_prefetch_map(&maps.tree_k);
        tma_prefetch_map(&maps.tree_v);
    }
    if (warp == kQkWarp) tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // The inputs may come from the previous kernel of the stream.
    pdl_wait_prior_grid();
    // The combine kernel may launch now: it waits for this grid before it
    // reads any partial or writes any output.
    pdl_launch_dependents();
    // 256 x 216 + 128 x 72 = 384 x 168, the registers the block launched with
    // (the host refuses to launch a build that uses any other count).
    if (warp >= kSoftmaxWarps) {
        setmaxnreg_dec<kOtherRegs>();
        if (warp == kProducerWarp)
            producer_loop<D, kPaged>(maps, L, a, sbase, bars, items_s, abort);
        else if (warp == kQkWarp)
            qk_loop<D>(a, sbase, bars, items_s, tmem, abort);
        else if (warp == kPvWarp)
            pv_loop<D>(a, smem, sbase, bars, items_s, tmem, abort);
        else if (warp == kVProducerWarp)
            v_producer_loop<D, kPaged>(maps, L, a, sbase, bars, items_s, abort);
    } else {
        setmaxnreg_inc<kSoftmaxRegs>();
        softmax_loop<D>(maps, L, a, smem, bars, items_s, reinterpret_cast<float *>(smem + C::hand_off),
                        reinterpret_cast<float *>(smem + C::xchg_off), tmem, abort);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kQkWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D, bool kPaged>
cudaError_t launch_d(const Layout &L, const AttnMaps &m, const AttnArgs &a, cudaStream_t s) {
    using C = AttnCfg<D>;
    static_assert(C::smem_request <= 227 * 1024, "shared memory budget");
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        // setmaxnreg hands out exactly the registers the block launched with;
        // a build with another per-thread count would make it wait forever.
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, tree_attention_kernel<D, kPaged>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(tree_attention_kernel<D, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::smem_request);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::smem_request;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin("tree_attention", s);
    e = cudaLaunchKernelEx(&cfg, tree_attention_kernel<D, kPaged>, m, L, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(s);
    return e;
}

}  // namespace

cudaError_t launch_tree_attention(const Layout &L, const AttnMaps &m, const AttnArgs &a, cudaStream_t s) {
    if (a.page_lg >= 0) return L.D == 128 ? launch_d<128, true>(L, m, a, s) : launch_d<64, true>(L, m, a, s);
    return L.D == 128 ? launch_d<128, false>(L, m, a, s) : launch_d<64, false>(L, m, a, s);
}

}  // namespace jf
