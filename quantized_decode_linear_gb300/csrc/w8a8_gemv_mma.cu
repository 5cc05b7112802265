// W8A8 decode GEMV for small token counts (w8a8_decode.rs fn w8a8_gemv;
// segment routing from W8a8Weight::boundaries; scale layouts from enum
// W8a8Scale).  HBM-bound: every weight byte is read once, 16 bytes per
// thread per load, evict-first in L2.
//
//   y[m, j] = sum_kb Sa(m, kb) Sw(j, kb) sum_{k in kb} dec(q[m,k]) dec(W[j,k])
//
// Work decomposition
//   CTA   = 8 warps = 128 consecutive output rows (weight rows) x a K range of
//           whole 128-blocks.  The K ranges of the CTAs of one cluster
//           (cluster dims 1 x split) tile K; the cluster reduces its partial
//           sums through distributed shared memory in a fixed order, so the
//           result does not depend on scheduling.
//   warp  = 16 weight rows.  Each 64-wide K chunk is one pair of
//           m16n8k32 e4m3 MMAs per 8 tokens (weights as the 16-row A operand,
//           tokens as the 8-column B operand), f32 accumulators.
//   K permutation: thread (g = lane/4, t = lane%4) loads 16 contiguous bytes
//           of weight rows g and g+8 and of token g at offset 16 t of the chunk.
//           The MMA's K index is permuted identically for A and B, which
//           leaves the dot product unchanged.
//   Scales: the MMA accumulates one 128-block; the block's partial sums are
//           then folded into f32 totals (Block128: times sa[m,kb] sw[j/128,kb];
//           PerRow: plain sum, scaled once at the end).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "qdl_internal.cuh"

namespace cg = cooperative_groups;

namespace qdl {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerCta = kWarps * 16;
constexpr int kDepth = 4;  // 64-wide K chunks in flight per warp

template <int NT, bool kBlock>
__global__ void __launch_bounds__(256, 2) w8a8_gemv_mma_kernel(W8A8Args a) {
    __shared__ float red[NT * 8][kRowsPerCta];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t row0 = blockIdx.x * kRowsPerCta + warp * 16;
    const uint32_t split = gridDim.y, sidx = blockIdx.y;
    const uint32_t kb0 = (a.kb * sidx) / split, kb1 = (a.kb * (sidx + 1)) / split;
    const uint64_t policy = policy_evict_first();

    // segment of this warp's 16 rows (never straddles: segment sizes other
    // than the last are multiples of 16)
    const uint8_t *wseg;
    const float *sseg;
    uint32_t lrow0;
    if (row0 < a.n1) {
        wseg = a.w0; sseg = a.sw0; lrow0 = row0;
    } else if (row0 < a.n2) {
        wseg = a.w1; sseg = a.sw1; lrow0 = row0 - a.n1;
    } else {
        wseg = a.w2; sseg = a.sw2; lrow0 = row0 - a.n2;
    }
    const bool warp_ok = row0 < a.n;  // else every row of the warp is past N
    const bool ok0 = row0 + g < a.n, ok1 = row0 + g + 8 < a.n;
    const uint8_t *wp0 = wseg + (size_t)(lrow0 + g) * a.k + 16 * t;
    const uint8_t *wp1 = wseg + (size_t)(lrow0 + g + 8) * a.k + 16 * t;

    const uint8_t *ap[NT];
    bool aok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint32_t tok = nt * 8 + g;
        aok[nt] = tok < a.m;
        ap[nt] = a.q + (size_t)(aok[nt] ? tok : 0) * a.k + 16 * t;
    }

    float total[NT][4], acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) total[nt][i] = acc[nt][i] = 0.0f;

    const uint32_t c0 = kb0 * 2, c1 = kb1 * 2;  // 64-wide chunks
    uint4 wb[kDepth][2];
    uint4 ab[kDepth][NT];
    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
        const uint32_t c = c0 + i;
        const bool in = c < c1;
        wb[i][0] = (in && ok0) ? ld_stream_v4(wp0 + c * 64, policy) : zero;
        wb[i][1] = (in && ok1) ? ld_stream_v4(wp1 + c * 64, policy) : zero;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ab[i][nt] = (in && aok[nt]) ? ld_ro_v4(ap[nt] + c * 64) : zero;
    }

    for (uint32_t cb = c0; cb < c1; cb += kDepth) {
#pragma unroll
        for (int i = 0; i < kDepth; ++i) {
            const uint32_t c = cb + i;
            if (c < c1) {
                const uint4 A0 = wb[i][0], A1 = wb[i][1];
                uint4 B[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) B[nt] = ab[i][nt];
                const uint32_t cn = c + kDepth;
                const bool in = cn < c1;
                wb[i][0] = (in && ok0) ? ld_stream_v4(wp0 + cn * 64, policy) : zero;
                wb[i][1] = (in && ok1) ? ld_stream_v4(wp1 + cn * 64, policy) : zero;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    ab[i][nt] = (in && aok[nt]) ? ld_ro_v4(ap[nt] + cn * 64) : zero;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_e4m3_16832(acc[nt], A0.x, A1.x, A0.y, A1.y, B[nt].x, B[nt].y);
                    mma_e4m3_16832(acc[nt], A0.z, A1.z, A0.w, A1.w, B[nt].z, B[nt].w);
                }
                if (c & 1) {  // end of a 128-block: fold the block's partial sums
                    const uint32_t kb = c >> 1;
                    if constexpr (kBlock) {
                        const float sw = warp_ok ? sseg[(size_t)(lrow0 >> 7) * a.kb + kb] : 0.0f;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint32_t tk = nt * 8 + 2 * t;
                            const float s0 = tk < a.m ? a.sa[(size_t)tk * a.kb + kb] * sw : 0.0f;
                            const float s1 = tk + 1 < a.m ? a.sa[(size_t)(tk + 1) * a.kb + kb] * sw : 0.0f;
                            total[nt][0] = fmaf(acc[nt][0], s0, total[nt][0]);
                            total[nt][1] = fmaf(acc[nt][1], s1, total[nt][1]);
                            total[nt][2] = fmaf(acc[nt][2], s0, total[nt][2]);
                            total[nt][3] = fmaf(acc[nt][3], s1, total[nt][3]);
                        }
                    } else {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int j = 0; j < 4; ++j) total[nt][j] += acc[nt][j];
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[nt][j] = 0.0f;
                }
            }
        }
    }

    if constexpr (!kBlock) {  // per-row scales: sa[token] * sw[row]
        const float sw0 = ok0 ? sseg[lrow0 + g] : 0.0f;
        const float sw1 = ok1 ? sseg[lrow0 + g + 8] : 0.0f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t tk = nt * 8 + 2 * t;
            const float s0 = tk < a.m ? a.sa[tk] : 0.0f;
            const float s1 = tk + 1 < a.m ? a.sa[tk + 1] : 0.0f;
            total[nt][0] *= s0 * sw0;
            total[nt][1] *= s1 * sw0;
            total[nt][2] *= s0 * sw1;
            total[nt][3] *= s1 * sw1;
        }
    }

    auto store = [&](uint32_t tok, uint32_t row, float v) {
        if (tok < a.m && row < a.n) {
            if (a.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)tok * a.ldc + row] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float *>(a.out)[(size_t)tok * a.ldc + row] = v;
        }
    };

    if (split == 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t tk = nt * 8 + 2 * t;
            store(tk, row0 + g, total[nt][0]);
            store(tk + 1, row0 + g, total[nt][1]);
            store(tk, row0 + g + 8, total[nt][2]);
            store(tk + 1, row0 + g + 8, total[nt][3]);
        }
        return;
    }

    // split-K across the cluster: partials to shared memory, then CTA r sums
    // rows [r*128/split, (r+1)*128/split) over all ranks in rank order.
    const int lr = warp * 16 + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int tk = nt * 8 + 2 * t;
        red[tk][lr] = total[nt][0];
        red[tk + 1][lr] = total[nt][1];
        red[tk][lr + 8] = total[nt][2];
        red[tk + 1][lr + 8] = total[nt][3];
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const uint32_t r_lo = (kRowsPerCta * sidx) / split, r_hi = (kRowsPerCta * (sidx + 1)) / split;
    const uint32_t span = r_hi - r_lo;
    for (uint32_t idx = threadIdx.x; idx < span * NT * 8; idx += blockDim.x) {
        const uint32_t tok = idx / span, lrow = r_lo + idx % span;
        float sum = 0.0f;
        for (uint32_t rk = 0; rk < split; ++rk) {
            const float *peer = cluster.map_shared_rank(&red[0][0], rk);
            sum += peer[tok * kRowsPerCta + lrow];
        }
        store(tok, blockIdx.x * kRowsPerCta + lrow, sum);
    }
    cluster.sync();
}

template <int NT, bool kBlock>
cudaError_t launch_nt(const W8A8Args &a, uint32_t split, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.n + kRowsPerCta - 1) / kRowsPerCta, split, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w8a8_gemv_mma_kernel<NT, kBlock>, a);
}

}  // namespace

// Split-K factor: the smallest power of two (<= 8, <= number of 128-blocks)
// that puts at least two CTAs on every SM.
static uint32_t choose_split(const W8A8Args &a) {
#ifdef QDL_TUNE_SPLIT
    if (QDL_TUNE_SPLIT > 0) return QDL_TUNE_SPLIT < a.kb ? QDL_TUNE_SPLIT : a.kb;
#endif
    const uint32_t tiles = (a.n + kRowsPerCta - 1) / kRowsPerCta;
    const uint32_t want = 2u * (uint32_t)device_sm_count();
    uint32_t split = 1;
    while (split < 8 && split * 2 <= a.kb && tiles * split < want) split *= 2;
    return split;
}

cudaError_t launch_w8a8_gemv_mma(const W8A8Args &a, int format, cudaStream_t s) {
    const uint32_t split = choose_split(a);
    const bool blk = format == QDL_SCALE_BLOCK128;
    if (a.m <= 8) return blk ? launch_nt<1, true>(a, split, s) : launch_nt<1, false>(a, split, s);
    return blk ? launch_nt<2, true>(a, split, s) : launch_nt<2, false>(a, split, s);
}

}  // namespace qdl
