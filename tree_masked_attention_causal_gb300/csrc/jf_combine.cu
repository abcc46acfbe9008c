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
// row o_s = O_s / l_s in fp16 plus (m_s, l_s) in fp32, with m in the exp2
// domain. The merged row is the log-sum-exp rescale:
//   O = sum_s w_s o_s / sum_s w_s,   w_s = 2^(m_s - M) l_s,   M = max_s m_s.
// The sums run in split order, so the result is deterministic.
//
// Grid (units, 128 / 8 rows), one warp per row, lane k holding d/32
// consecutive columns. The (m, l) of all splits and the O rows of up to 8
// splits are loaded in one round trip. The kernel is a programmatic
// dependent of the attention kernel: it validates the tree (inputs only)
// while that kernel runs, then waits for it before reading any partial or
// writing any output.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kCombineRowsPerBlock = 8;      // one warp per row
constexpr int kCombineThreads = 32 * kCombineRowsPerBlock;
constexpr int kCombineBatch = 8;             // splits whose loads are issued together

template <int D>
__global__ void __launch_bounds__(kCombineThreads) split_combine_kernel(const Layout L, const AttnArgs a) {
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
    bad = __syncthreads_or(bad);
    pdl_wait_prior_grid();          // the attention grid is complete from here on
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y * kCombineRowsPerBlock + warp;
    const int node = qt * L.NB + r / L.G;
    if (node >= L.Nmax) return;
    const int head = kh * L.G + r % L.G;
    constexpr int E = D / 32;   // columns per lane
    __nv_bfloat16 *dst = a.out + (((size_t)b * L.Nmax + node) * L.Hq + head) * D + lane * E;
    if (bad) {
        if (kh == 0 && qt == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_status(a.status, JF_STATUS_BAD_TREE);
        const uint32_t nan2 = 0x7FC07FC0u;
        if constexpr (E == 4)
            *reinterpret_cast<uint2 *>(dst) = make_uint2(nan2, nan2);
        else
            *reinterpret_cast<uint32_t *>(dst) = nan2;
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
    const float2 *ml = reinterpret_cast<const float2 *>(a.ws + L.ml_off);
    const __half *op = reinterpret_cast<const __half *>(a.ws + L.opart_off);
    constexpr float kNegInf = -__builtin_huge_valf();
    // (m_s, l_s): lane s holds split s (splits past 32 are folded in below)
    float2 mine = make_float2(kNegInf, 0.f);
    if (lane < ns) mine = __ldcg(&ml[(size_t)slot_of(lane) * kRows + r]);
    float M = mine.x;
    for (int s = 32 + lane; s < ns; s += 32) M = fmaxf(M, __ldcg(&ml[(size_t)slot_of(s) * kRows + r]).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == kNegInf) M = 0.f;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float Lsum = 0.f;
    for (int s0 = 0; s0 < ns; s0 += kCombineBatch) {
        uint32_t v[kCombineBatch][E / 2];           // fp16 pairs
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {    // all loads of the batch first
            const int s = s0 + k;
            if (s < ns) {
                const __half *src = op + ((size_t)slot_of(s) * kRows + r) * D + lane * E;
                if constexpr (E == 4) {
                    const uint2 x = __ldcg(reinterpret_cast<const uint2 *>(src));
                    v[k][0] = x.x;
                    v[k][1] = x.y;
                } else {
                    v[k][0] = __ldcg(reinterpret_cast<const unsigned int *>(src));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {    // then the weighted sums, in split order
            const int s = s0 + k;
            if (s < ns) {
                const float2 mls = s < 32 ? make_float2(__shfl_sync(0xffffffffu, mine.x, s),
                                                        __shfl_sync(0xffffffffu, mine.y, s))
                                          : __ldcg(&ml[(size_t)slot_of(s) * kRows + r]);
                // the piece is O_s / l_s: its weight in the sum is 2^(m_s - M) l_s
                const float w = ex2_approx(mls.x - M) * mls.y;
                Lsum += w;
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&v[k][e]));
                    acc[2 * e] += w * f.x;
                    acc[2 * e + 1] += w * f.y;
                }
            }
        }
    }
    const float inv = 1.0f / Lsum;
    if constexpr (E == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                     pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
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
