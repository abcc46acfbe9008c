// jf_combine.cu - merge of the split-KV partials of tree attention.
//
// A work unit whose keys were split over several CTAs has, per split s, an
// unnormalised fp32 row O_s plus (m_s, l_s), with m in the exp2 domain. The
// merged row is the log-sum-exp rescale:
//   O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
// The sums run in split order, so the result is deterministic.
//
// The merge is spread over the whole GPU: grid (units, 256 / 8 rows), one
// warp per row, lane k holding d/32 consecutive columns. The (m, l) of all
// splits and the O rows of up to 8 splits are loaded in one round trip.
// The kernel is a programmatic dependent of the attention kernel: it
// launches while that kernel runs and waits for it before reading any
// partial.
#include "jf_common.cuh"

namespace jf {
namespace {

constexpr int kCombineRowsPerBlock = 8;      // one warp per row
constexpr int kCombineThreads = 32 * kCombineRowsPerBlock;
constexpr int kCombineBatch = 8;             // splits whose loads are issued together

template <int D>
__global__ void __launch_bounds__(kCombineThreads) split_combine_kernel(const Layout L, const AttnArgs a) {
    pdl_wait_prior_grid();
    const int q = blockIdx.x;
    const QTile qi = reinterpret_cast<const QTile *>(a.ws + L.qtab_off)[q];
    const int ns = qi.n_splits, base = qi.slot_base;
    if (ns <= 1) return;
    const int b = q / (L.Hkv * L.QT);
    const int rem = q - b * (L.Hkv * L.QT);
    const int kh = rem / L.QT, qt = rem - kh * L.QT;
    const SeqInfo si = reinterpret_cast<const SeqInfo *>(a.ws + L.seq_off)[b];
    if (si.bad) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y * kCombineRowsPerBlock + warp;
    const int node = qt * L.NB + r / L.G;
    if (node >= si.n_nodes) return;
    const int head = kh * L.G + r % L.G;
    const float2 *ml = reinterpret_cast<const float2 *>(a.ws + L.ml_off);
    const float *op = reinterpret_cast<const float *>(a.ws + L.opart_off);
    constexpr int E = D / 32;   // columns per lane
    constexpr float kNegInf = -__builtin_huge_valf();
    // (m_s, l_s): lane s holds split s (splits past 32 are folded in below)
    float2 mine = make_float2(kNegInf, 0.f);
    if (lane < ns) mine = __ldcg(&ml[(size_t)(base + lane) * kRows + r]);
    float M = mine.x;
    for (int s = 32 + lane; s < ns; s += 32) M = fmaxf(M, __ldcg(&ml[(size_t)(base + s) * kRows + r]).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == kNegInf) M = 0.f;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float Lsum = 0.f;
    for (int s0 = 0; s0 < ns; s0 += kCombineBatch) {
        float v[kCombineBatch][E];
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {    // all loads of the batch first
            const int s = s0 + k;
            if (s < ns) {
                const float *src = op + ((size_t)(base + s) * kRows + r) * D + lane * E;
                if constexpr (E == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
                    v[k][0] = x.x; v[k][1] = x.y; v[k][2] = x.z; v[k][3] = x.w;
                } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
                    v[k][0] = x.x; v[k][1] = x.y;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {    // then the weighted sums, in split order
            const int s = s0 + k;
            if (s < ns) {
                const float2 mls = s < 32 ? make_float2(__shfl_sync(0xffffffffu, mine.x, s),
                                                        __shfl_sync(0xffffffffu, mine.y, s))
                                          : __ldcg(&ml[(size_t)(base + s) * kRows + r]);
                const float w = ex2_approx(mls.x - M);
                Lsum += w * mls.y;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] += w * v[k][e];
            }
        }
    }
    const float inv = 1.0f / Lsum;
    __nv_bfloat16 *dst = a.out + (((size_t)b * L.Nmax + node) * L.Hq + head) * D + lane * E;
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
