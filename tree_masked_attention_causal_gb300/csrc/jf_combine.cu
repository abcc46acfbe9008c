// jf_combine.cu - the kernel that follows tree attention: tree validation,
// the NaN rows of malformed sequences, and the merge of split-KV partials.
//
// Validation follows the tree's definition (node 0 is the root, parent[0] =
// -1, every other node's parent comes earlier, 0 <= parent[i] < i), plus the
// ranges of n_nodes and prefix_lens. Every output row of a sequence that
// fails it becomes NaN and JF_STATUS_BAD_TREE is raised; the attention kernel
// has computed those rows without checking, and they are overwritten here.
//
// A work unit whose keys were split over several CTAs has, per split s, a
// row o_s = O_s / l_s in fp16, scaled by 2^-e per half row so that fp16
// holds any bf16 magnitude, plus (m_s, l_s, e) in fp32, with m in the exp2
// domain. The merged row is the log-sum-exp rescale:
//   O = sum_s w_s 2^e o_s / sum_s w_s,   w_s = 2^(m_s - M) l_s,   M = max_s m_s.
// The sums run in split order, so the result is deterministic.
//
// Grid (units, 128 / 16 rows), two rows per warp (16 lanes each, lane k
// holding d/16 consecutive columns), so that every block of a work unit of
// the benchmark shape is resident in one wave. The (m, l) of all splits and
// the O rows of the first 4 splits are requested in one round trip. The kernel is a programmatic
// dependent of the attention kernel: it validates the tree (inputs only)
// while that kernel runs, then waits for it before reading any partial or
// writing any output.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kCombineRowsPerBlock = 16;     // two rows per warp, 16 lanes per row
constexpr int kCombineThreads = 256;
constexpr int kCombineBatch = 4;             // splits whose loads are issued together
constexpr int kGroup = 16;                   // lanes per row

// Loads of E consecutive fp16 (E = 8: 16 B, E = 4: 8 B).
template <int E>
struct HalfVec;
template <>
struct HalfVec<8> {
    uint4 v;
    __device__ void load(const __half *p) { v = __ldcg(reinterpret_cast<const uint4 *>(p)); }
    __device__ uint32_t word(int k) const { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; }
};
template <>
struct HalfVec<4> {
    uint2 v;
    __device__ void load(const __half *p) { v = __ldcg(reinterpret_cast<const uint2 *>(p)); }
    __device__ uint32_t word(int k) const { return k == 0 ? v.x : v.y; }
};

template <int D>
__global__ void __launch_bounds__(kCombineThreads, 4) split_combine_kernel(const Layout L, const AttnArgs a) {
    const int q = blockIdx.x;
    const int b = q / (L.Hkv * L.QT);
    const int rem = q - b * (L.Hkv * L.QT);
    const int kh = rem / L.QT, qt = rem - kh * L.QT;
    // Validate sequence b: one node per thread (Nmax <= blockDim).
    const int P = a.prefix_lens[b], n = a.n_nodes[b];
    const int i = threadIdx.x;
    bool bad = !seq_valid(P, n, L);
    if (!bad && i < n) {
        const int p = a.parents[(size_t)b * L.Nmax + i];
        bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
    }
    if (!bad && a.page_lg >= 0) {                          // every page the prefix uses is a real page
        const int used = (P + (1 << a.page_lg) - 1) >> a.page_lg;
        for (int j = i; !bad && j < used; j += blockDim.x) {
            const int ph = a.block_table[(size_t)b * a.pages_per_seq + j];
            bad = ph < 0 || ph >= a.num_pages;
        }
    }
    bad = __syncthreads_or(bad);
    pdl_wait_prior_grid();          // the attention grid is complete from here on
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane & (kGroup - 1);                     // lane within the row's group
    const unsigned gmask = (lane < kGroup) ? 0x0000FFFFu : 0xFFFF0000u;
    const int r = blockIdx.y * kCombineRowsPerBlock + warp * 2 + (lane >> 4);
    const int node = (qt << L.lgNB) + (r >> L.lgG);
    if (node >= L.Nmax) return;                            // whole 16-lane groups leave together
    const int head = (kh << L.lgG) + (r & (L.G - 1));
    constexpr int E = D / kGroup;                          // columns per lane
    __nv_bfloat16 *dst = a.out + (((size_t)b * L.Nmax + node) * L.Hq + head) * D + g * E;
    if (bad) {
        if (kh == 0 && qt == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_status(a.status, JF_STATUS_BAD_TREE);
        const uint32_t nan2 = 0x7FC07FC0u;
        if constexpr (E == 8)
            *reinterpret_cast<uint4 *>(dst) = make_uint4(nan2, nan2, nan2, nan2);
        else
            *reinterpret_cast<uint2 *>(dst) = make_uint2(nan2, nan2);
        return;
    }
    if (node >= n || unit_tiles(P, n, qt, L) == 0) return;
    const QTile qi = reinterpret_cast<const QTile *>(a.ws + L.qtab_off)[q];
    const int ns = qi.n_splits;
    if (ns <= 1) return;
    // The attention kernel records the plan of every unit with work; one that
    // aborted (JF_STATUS_TIMEOUT) may not have: never follow slots outside
    // the partial buffers.
    if (qi.c_first < 0 || 2 * (qi.c_first + ns) > L.max_pieces) return;
    // split s sits in slot 2c + 1 at c = c_first when the unit is not that
    // CTA's first item, else in slot 2c, c = c_first + s
    auto slot_of = [&](int sidx) { return 2 * (qi.c_first + sidx) + ((sidx == 0 && !qi.first_item) ? 1 : 0); };
    const float4 *ml = reinterpret_cast<const float4 *>(a.ws + L.ml_off);   // (m, l, e0, e1)
    const __half *op = reinterpret_cast<const __half *>(a.ws + L.opart_off);
    constexpr float kNegInf = -__builtin_huge_valf();
    // The first batch of O pieces is requested together with (m, l).
    HalfVec<E> v[kCombineBatch];
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k)
        if (k < ns) v[k].load(op + ((size_t)slot_of(k) * kRows + r) * D + g * E);
    // (m_s, l_s, e): lane g of the group holds split g (more are folded in
    // below); e is the exponent of the half row that holds this lane's columns
    const int half = (g * E) / (D / 2);
    float4 rec = make_float4(kNegInf, 0.f, 0.f, 0.f);
    if (g < ns) rec = __ldcg(&ml[(size_t)slot_of(g) * kRows + r]);
    float M = rec.x;
    for (int s = kGroup + g; s < ns; s += kGroup) M = fmaxf(M, __ldcg(&ml[(size_t)slot_of(s) * kRows + r]).x);
#pragma unroll
    for (int o = kGroup / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(gmask, M, o));
    if (M == kNegInf) M = 0.f;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float Lsum = 0.f;
    const int gbase = lane & kGroup;                       // first lane of this row's group
    for (int s0 = 0; s0 < ns; s0 += kCombineBatch) {
        if (s0 > 0) {
#pragma unroll
            for (int k = 0; k < kCombineBatch; ++k)
                if (s0 + k < ns) v[k].load(op + ((size_t)slot_of(s0 + k) * kRows + r) * D + g * E);
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {          // weighted sums, in split order
            const int s = s0 + k;
            if (s < ns) {
                float4 r4;
                if (s < kGroup) {
                    r4.x = __shfl_sync(gmask, rec.x, gbase + s);
                    r4.y = __shfl_sync(gmask, rec.y, gbase + s);
                    r4.z = __shfl_sync(gmask, rec.z, gbase + s);
                    r4.w = __shfl_sync(gmask, rec.w, gbase + s);
                } else {
                    r4 = __ldcg(&ml[(size_t)slot_of(s) * kRows + r]);
                }
                // the piece is O_s / (l_s 2^e): its weight in the sum is
                // 2^(m_s - M) l_s, and its values count 2^e times
                const float w = ex2_approx(r4.x - M) * r4.y;
                Lsum += w;
                const int eh = __float2int_rz(half ? r4.w : r4.z);
                const float we = w * __int_as_float((127 + eh) << 23);            // w * 2^e, exact
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    const uint32_t h2 = v[k].word(e);
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                    acc[2 * e] += we * f.x;
                    acc[2 * e + 1] += we * f.y;
                }
            }
        }
    }
    const float inv = 1.0f / Lsum;
    if constexpr (E == 8) {
        *reinterpret_cast<uint4 *>(dst) =
            make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                       pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
    } else {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                     pack_bf16x2(acc[2] * inv, acc[3] * inv));
    }
}

}  // namespace

cudaError_t launch_split_combine(const Layout &L, const AttnArgs &a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.n_qtiles, kRows / kCombineRowsPerBlock);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin("split_combine", s);
    cudaError_t e = L.D == 128 ? cudaLaunchKernelEx(&cfg, split_combine_kernel<128>, L, a)
                               : cudaLaunchKernelEx(&cfg, split_combine_kernel<64>, L, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    trace_end(s);
    return e;
}

}  // namespace jf
