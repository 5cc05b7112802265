// Activation quantisation to FP8 E4M3 (w8a8_decode.rs: w8a8_act_quant and
// w8a8_act_quant_silu; scale layout from W8a8Scale::act_scales_per_row).
//
//   s = absmax / 448            (IEEE binary32 division)
//   q = e4m3_rne_sat(act / s)   (IEEE division, then cvt.rn.satfinite)
//   act = x, or SiLU(gate) * up computed with the library's exp
//
// A group whose absmax is 0 stores s = 0 and the codes of its signed zeros.
// Every step is a correctly rounded binary32 operation, so codes and scales
// are reproducible bit for bit.
//
// Two kernels:
//   - per 128-group (Block128): one warp per group, 4 elements per lane,
//     absmax by warp shuffles; the grid covers rows x k/128 groups.
//   - per token row (PerRow): each row is split over a cluster of up to 8
//     CTAs; each thread keeps its elements in registers (UPT 16-byte units of
//     8 values), absmax by warp shuffles, shared memory and then distributed
//     shared memory across the cluster, then quantises from registers.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "qdl_internal.cuh"

namespace cg = cooperative_groups;

namespace qdl {
namespace {

template <bool kSilu>
__device__ __forceinline__ float act_value(uint32_t a_bits, uint32_t b_bits) {
    const float a = bf16_bits_to_f32(a_bits);
    if constexpr (kSilu) {
        return silu_mul(a, bf16_bits_to_f32(b_bits));
    } else {
        return a;
    }
}

__device__ __forceinline__ float quant_operand(float v, float scale) {
    return scale == 0.0f ? v : __fdiv_rn(v, scale);
}

// ---------------------------------------------------------------- Block128

// Programmatic launch overlap: let the next kernel (the GEMV) launch at once,
// so that its CTAs take SMs as the previous kernel's CTAs leave and start
// streaming their weights; then wait for the previous kernel, since the input
// comes from it and the scratch written here may still be read by it.  (The
// GEMV reads this kernel's output only after its own dependency wait, which
// returns when this grid has completed.)
__device__ __forceinline__ void dependent_launch_prologue() {
#if QDL_TUNE_EARLY_TRIGGER
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#else
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Zero out[0..rows)[0..zn) (row stride zldc) with the whole grid: chunks of 4
// columns (float4 stores where the rows allow), walked as (row, chunk) pairs
// from one division per thread.
__device__ __forceinline__ void zero_rows(const ActQuantArgs &a) {
    const bool vec = (reinterpret_cast<uintptr_t>(a.zout) % 16 == 0) && a.zldc % 4 == 0;
    const uint32_t cw = vec ? 4u : 1u;             // columns per chunk
    const uint32_t cpr = (a.zn + cw - 1) / cw;     // chunks per row
    const uint32_t nthreads = gridDim.x * blockDim.x, t = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t dr = nthreads / cpr, dc = nthreads % cpr;
    uint32_t r = t / cpr, c = t % cpr;
    while (r < a.rows) {
        float *row = a.zout + (size_t)r * a.zldc;
        const uint32_t col = c * cw;
        if (vec && col + 4 <= a.zn)
            *reinterpret_cast<float4 *>(row + col) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        else
            for (uint32_t i = col; i < col + cw && i < a.zn; ++i) row[i] = 0.0f;
        r += dr;
        c += dc;
        if (c >= cpr) {
            c -= cpr;
            ++r;
        }
    }
}

template <bool kSilu>
__global__ void __launch_bounds__(256) act_quant_g128_kernel(ActQuantArgs a) {
    dependent_launch_prologue();
    if (a.zout != nullptr) zero_rows(a);  // the whole grid zeroes the output rows
    const uint32_t groups_per_row = a.k / kKUnit;
    const uint32_t gid = blockIdx.x * 8 + (threadIdx.x >> 5);
    const uint32_t lane = threadIdx.x & 31;
    if (gid >= a.rows * groups_per_row) return;  // warp-uniform
    const uint32_t row = gid / groups_per_row;
    const uint32_t col = (gid % groups_per_row) * kKUnit + lane * 4;

    const uint2 xa = *reinterpret_cast<const uint2 *>(a.a + (size_t)row * a.lda + col);
    uint2 xb = make_uint2(0, 0);
    if constexpr (kSilu) xb = *reinterpret_cast<const uint2 *>(a.b + (size_t)row * a.ldb + col);

    float v[4];
    v[0] = act_value<kSilu>(xa.x & 0xFFFFu, xb.x & 0xFFFFu);
    v[1] = act_value<kSilu>(xa.x >> 16, xb.x >> 16);
    v[2] = act_value<kSilu>(xa.y & 0xFFFFu, xb.y & 0xFFFFu);
    v[3] = act_value<kSilu>(xa.y >> 16, xb.y >> 16);

    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = __fdiv_rn(amax, 448.0f);

    const uint32_t lo = cvt_e4m3x2(quant_operand(v[0], scale), quant_operand(v[1], scale));
    const uint32_t hi = cvt_e4m3x2(quant_operand(v[2], scale), quant_operand(v[3], scale));
    *reinterpret_cast<uint32_t *>(a.q + (size_t)row * a.k + col) = lo | (hi << 16);
    if (lane == 0) a.s[(size_t)row * groups_per_row + col / kKUnit] = scale;
}

// ---------------------------------------------------------------- PerRow

// One row is split over a cluster of C CTAs (blockIdx.x = rank): each CTA
// keeps its part of the row in registers (UPT 16-byte units of 8 values per
// thread), reduces its absmax by warp shuffles and shared memory, and the
// cluster combines the C partial maxima through distributed shared memory
// (max is exact and order-free, so every rank gets the same absmax).
template <bool kSilu, int UPT>
__global__ void __launch_bounds__(1024) act_quant_row_kernel(ActQuantArgs a) {
    __shared__ float warp_max[32];
    __shared__ float cta_max;
    dependent_launch_prologue();
    const uint32_t row = blockIdx.y;
    if (a.zout != nullptr) {  // the row's ranks zero its output row
        const uint32_t stride = gridDim.x * blockDim.x;
        for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < a.zn; c += stride)
            a.zout[(size_t)row * a.zldc + c] = 0.0f;
    }
    const uint32_t nrank = gridDim.x, rank = blockIdx.x;
    const uint32_t units = a.k / 8;
    const uint32_t per = (units + nrank - 1) / nrank;
    const uint32_t u0 = rank * per, u1 = u0 + per < units ? u0 + per : units;
    const uint16_t *xa = a.a + (size_t)row * a.lda;
    const uint16_t *xb = kSilu ? a.b + (size_t)row * a.ldb : nullptr;

    float v[UPT][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const uint32_t u = u0 + threadIdx.x + i * blockDim.x;
        if (u < u1) {
            const uint4 pa = *reinterpret_cast<const uint4 *>(xa + u * 8);
            uint4 pb = make_uint4(0, 0, 0, 0);
            if constexpr (kSilu) pb = *reinterpret_cast<const uint4 *>(xb + u * 8);
            const uint32_t wa[4] = {pa.x, pa.y, pa.z, pa.w};
            const uint32_t wb[4] = {pb.x, pb.y, pb.z, pb.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[i][2 * j] = act_value<kSilu>(wa[j] & 0xFFFFu, wb[j] & 0xFFFFu);
                v[i][2 * j + 1] = act_value<kSilu>(wa[j] >> 16, wb[j] >> 16);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t nwarps = blockDim.x >> 5;
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    if (warp == 0) {
        amax = lane < nwarps ? warp_max[lane] : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) cta_max = amax;
    }
    if (nrank > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every rank's cta_max is written
        if (warp == 0) {
            float m = lane < nrank ? *cluster.map_shared_rank(&cta_max, lane) : 0.0f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) warp_max[0] = m;
        }
        cluster.sync();  // no rank leaves or overwrites while others still read its cta_max
    } else {
        __syncthreads();
        if (threadIdx.x == 0) warp_max[0] = cta_max;
    }
    __syncthreads();
    const float scale = __fdiv_rn(warp_max[0], 448.0f);

    uint8_t *qrow = a.q + (size_t)row * a.k;
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
        const uint32_t u = u0 + threadIdx.x + i * blockDim.x;
        if (u < u1) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[j] = cvt_e4m3x2(quant_operand(v[i][2 * j], scale),
                                  quant_operand(v[i][2 * j + 1], scale));
            *reinterpret_cast<uint2 *>(qrow + u * 8) =
                make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
        }
    }
    if (rank == 0 && threadIdx.x == 0) a.s[row] = scale;
}

template <typename Kernel>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, cudaStream_t s, const ActQuantArgs &a,
                       uint32_t cluster_x = 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (QDL_TUNE_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Ranks per row: enough CTAs to cover the SMs about twice (up to 8, the
// portable cluster size), but at least 256 units of 8 values per rank; short
// rows stay in one CTA, where the cluster barriers would cost more than the
// split saves.
template <bool kSilu>
cudaError_t launch_row(const ActQuantArgs &a, cudaStream_t s) {
    const uint32_t units = a.k / 8;
    const uint32_t want = (2u * (uint32_t)device_sm_count() + a.rows - 1) / a.rows;
    uint32_t ranks = want < 1 ? 1 : want > 8 ? 8 : want;
    while (ranks > 1 && units / ranks < 256) --ranks;
    const uint32_t per = (units + ranks - 1) / ranks;
    uint32_t threads = per < 1024 ? ((per + 31) / 32) * 32 : 1024;
    if (threads < 64) threads = 64;
    const uint32_t upt = (per + threads - 1) / threads;
    dim3 grid(ranks, a.rows), block(threads);
    if (upt <= 1) return launch_pdl(act_quant_row_kernel<kSilu, 1>, grid, block, s, a, ranks);
    if (upt <= 2) return launch_pdl(act_quant_row_kernel<kSilu, 2>, grid, block, s, a, ranks);
    if (upt <= 4) return launch_pdl(act_quant_row_kernel<kSilu, 4>, grid, block, s, a, ranks);
    return launch_pdl(act_quant_row_kernel<kSilu, 8>, grid, block, s, a, ranks);
}

template <bool kSilu>
cudaError_t launch_g128(const ActQuantArgs &a, cudaStream_t s) {
    const uint32_t groups = a.rows * (a.k / kKUnit);
    return launch_pdl(act_quant_g128_kernel<kSilu>, dim3((groups + 7) / 8), dim3(256), s, a);
}

}  // namespace

cudaError_t launch_act_quant(const ActQuantArgs &a, int format, bool silu, cudaStream_t s) {
    if (format == QDL_SCALE_PER_ROW) return silu ? launch_row<true>(a, s) : launch_row<false>(a, s);
    return silu ? launch_g128<true>(a, s) : launch_g128<false>(a, s);
}

}  // namespace qdl
