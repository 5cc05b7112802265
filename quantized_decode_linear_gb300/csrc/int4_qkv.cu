// AWQ INT4 fused Q/K/V projection (fused_int4_qkv.rs: fused_int4_qkv_q,
// fused_int4_qkv_k, fused_int4_qkv_v, unpack_awq_qkv, QKV_AWQ_SHIFTS).
// One launch covers all three projections.
//
// Arithmetic.  With w = (nib - z) s per group of `group` K values, the
// product is regrouped so that the tensor cores see exact small integers:
//   y[m, c] = sum_g s[g,c] ( sum_{k in g} x~[m,k] nib[k,c]
//                            - z[g,c] sum_{k in g} x~[m,k] )
// x~ = x rounded to f16 (used in both terms, so the identity is exact in
// x~); nib is exact in f16; products are exact in the f32 accumulators.
// The only approximation is x -> x~, |x~ - x| <= 2^-11 |x|, which bounds the
// error by 2^-11 sum_k |x w|.  sum_k x~ per group comes from one extra MMA
// against an all-ones A operand, so it sees the same x~.
//
// Unpacking.  AWQ stores the 8 columns of a word at shifts
// {0,16,4,20,8,24,12,28}: physical nibble p holds column {0,2,4,6,1,3,5,7}[p].
// For two consecutive K rows k, k+1 of the same word column, a byte permute
// puts the low halves (or high halves) of both words side by side; then
// (X >> 4j) & 0x000F000F | 0x64006400 is the f16 pair (1024 + nib(k),
// 1024 + nib(k+1)) of one column, and one f16x2 subtraction of 1024 leaves
// the exact nibbles, paired along K as the MMA operand wants.  This is the
// published AWQ / Marlin-style interleave-to-f16 conversion (the 4-bit value
// ORed into the mantissa of 1024.0 in f16), implemented from its description.
//
// Tiling.  A warp owns 128 columns (16 per 4-lane group: two packed words)
// as eight m16n8k16 tiles (columns as the MMA's M, tokens as N, K = 16).
// Lane (g, t) loads K rows k0+4t .. k0+4t+3 of its two word columns; the
// MMA's K index is permuted identically for A and B.  The CTA's 8 warps
// split the CTA's K range by whole groups; the cluster (1 x split CTAs)
// splits K further.  Partial sums are reduced in shared memory and then
// across the cluster in a fixed order.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "qdl_internal.cuh"

namespace cg = cooperative_groups;

namespace qdl {
namespace {

constexpr int kWarps = 8;
constexpr int kCols = 128;  // columns per CTA (one warp's width)

// column (within the warp's 128) held by MMA tile i, row r of the tile
__device__ __forceinline__ uint32_t tile_col(int i, int r) {
    const int word_col = 2 * (r & 7) + (r >> 3);
    const int in_word = i < 4 ? 2 * i : 2 * (i - 4) + 1;
    return 8 * word_col + in_word;
}

__device__ __forceinline__ uint32_t nib_pair(uint32_t perm, int j) {
    const uint32_t v = ((perm >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&v), __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int NT>
__global__ void __launch_bounds__(256, 1) int4_qkv_kernel(Int4Args a) {
    extern __shared__ float smem[];  // [kWarps][NT*8][kCols] then [NT*8][kCols]
    float *red = smem;
    float *part = smem + kWarps * NT * 8 * kCols;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    // projection and column tile of this CTA
    uint32_t tile = blockIdx.x;
    const uint32_t *qw;
    const float *sc, *zr;
    float *out;
    uint32_t n;
    if (tile < a.tiles_q) {
        qw = a.qw0; sc = a.sc0; zr = a.zr0; out = a.out0; n = a.nq;
    } else if (tile < a.tiles_q + a.tiles_kv) {
        tile -= a.tiles_q;
        qw = a.qw1; sc = a.sc1; zr = a.zr1; out = a.out1; n = a.nkv;
    } else {
        tile -= a.tiles_q + a.tiles_kv;
        qw = a.qw2; sc = a.sc2; zr = a.zr2; out = a.out2; n = a.nkv;
    }
    const uint32_t npk = n / 8;
    const uint32_t col0 = tile * kCols;                // first column of the CTA
    const uint32_t wc0 = col0 / 8 + 2 * g;             // this lane's first word column
    const bool okw0 = wc0 < npk, okw1 = wc0 + 1 < npk;

    // K range of this warp, in groups
    const uint32_t split = gridDim.y;
    const uint32_t workers = split * kWarps, wid = blockIdx.y * kWarps + warp;
    const uint32_t gb0 = (a.groups * wid) / workers, gb1 = (a.groups * (wid + 1)) / workers;
    const uint32_t steps_per_group = a.group / 16;

    const uint64_t policy = policy_evict_first();
    const float *xrow[NT];
    bool xok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint32_t tok = nt * 8 + g;
        xok[nt] = tok < a.m;
        xrow[nt] = a.x + (size_t)(xok[nt] ? tok : 0) * a.k + 4 * t;
    }

    float total[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) total[nt][i][j] = 0.0f;

    auto load_words = [&](uint32_t k0, uint2 (&w)[4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t *p = qw + (size_t)(k0 + 4 * t + r) * npk + wc0;
            if (a.vec2) {
                w[r] = okw0 ? ld_stream_v2(p, policy) : make_uint2(0, 0);
            } else {
                w[r].x = okw0 ? ld_stream_u32(p, policy) : 0u;
                w[r].y = okw1 ? ld_stream_u32(p + 1, policy) : 0u;
            }
        }
    };

    for (uint32_t grp = gb0; grp < gb1; ++grp) {
        float acc[NT][8][4], ones[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[nt][i][j] = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) ones[nt][j] = 0.0f;
        }
        const uint32_t kg = grp * a.group;
        uint2 wcur[4], wnext[4];
        load_words(kg, wcur);
        for (uint32_t s = 0; s < steps_per_group; ++s) {
            const uint32_t k0 = kg + 16 * s;
            if (s + 1 < steps_per_group) load_words(k0 + 16, wnext);
            uint32_t b[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float4 xv = xok[nt] ? __ldg(reinterpret_cast<const float4 *>(xrow[nt] + k0))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                b[nt][0] = f16x2(xv.x, xv.y);
                b[nt][1] = f16x2(xv.z, xv.w);
            }
            // byte permutes: rows (4t, 4t+1) and (4t+2, 4t+3), word columns 0/1
            const uint32_t p00 = __byte_perm(wcur[0].x, wcur[1].x, 0x5410);
            const uint32_t q00 = __byte_perm(wcur[0].x, wcur[1].x, 0x7632);
            const uint32_t p01 = __byte_perm(wcur[0].y, wcur[1].y, 0x5410);
            const uint32_t q01 = __byte_perm(wcur[0].y, wcur[1].y, 0x7632);
            const uint32_t p10 = __byte_perm(wcur[2].x, wcur[3].x, 0x5410);
            const uint32_t q10 = __byte_perm(wcur[2].x, wcur[3].x, 0x7632);
            const uint32_t p11 = __byte_perm(wcur[2].y, wcur[3].y, 0x5410);
            const uint32_t q11 = __byte_perm(wcur[2].y, wcur[3].y, 0x7632);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = i & 3;
                const uint32_t a0 = nib_pair(i < 4 ? p00 : q00, j);  // row g,   k 4t..4t+1
                const uint32_t a1 = nib_pair(i < 4 ? p01 : q01, j);  // row g+8, k 4t..4t+1
                const uint32_t a2 = nib_pair(i < 4 ? p10 : q10, j);  // row g,   k 4t+2..4t+3
                const uint32_t a3 = nib_pair(i < 4 ? p11 : q11, j);  // row g+8, k 4t+2..4t+3
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16_16816(acc[nt][i], a0, a1, a2, a3, b[nt][0], b[nt][1]);
            }
            const uint32_t one = 0x3C003C00u;  // f16 pair (1, 1)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16_16816(ones[nt], one, one, one, one, b[nt][0], b[nt][1]);
#pragma unroll
            for (int r = 0; r < 4; ++r) wcur[r] = wnext[r];
        }
        // fold the group: total += s (acc - z sum_x)
        const float *scg = sc + (size_t)grp * n + col0 + 16 * g;
        const float *zrg = zr + (size_t)grp * n + col0 + 16 * g;
        float scv[16], zrv[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const bool ok = (v < 2) ? okw0 : okw1;
            const float4 s4 = ok ? __ldg(reinterpret_cast<const float4 *>(scg) + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 z4 = ok ? __ldg(reinterpret_cast<const float4 *>(zrg) + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            scv[4 * v] = s4.x; scv[4 * v + 1] = s4.y; scv[4 * v + 2] = s4.z; scv[4 * v + 3] = s4.w;
            zrv[4 * v] = z4.x; zrv[4 * v + 1] = z4.y; zrv[4 * v + 2] = z4.z; zrv[4 * v + 3] = z4.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int cw = i < 4 ? 2 * i : 2 * (i - 4) + 1;  // column within the word
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float s0 = ones[nt][0], s1 = ones[nt][1];  // sum_x of tokens 2t, 2t+1
                total[nt][i][0] += scv[cw] * (acc[nt][i][0] - zrv[cw] * s0);
                total[nt][i][1] += scv[cw] * (acc[nt][i][1] - zrv[cw] * s1);
                total[nt][i][2] += scv[8 + cw] * (acc[nt][i][2] - zrv[8 + cw] * s0);
                total[nt][i][3] += scv[8 + cw] * (acc[nt][i][3] - zrv[8 + cw] * s1);
            }
        }
    }

    // warp partials -> shared memory [warp][token][column]
    float *wred = red + (size_t)warp * NT * 8 * kCols;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int tk = nt * 8 + 2 * t;
            const uint32_t c0 = tile_col(i, g), c1 = tile_col(i, g + 8);
            wred[tk * kCols + c0] = total[nt][i][0];
            wred[(tk + 1) * kCols + c0] = total[nt][i][1];
            wred[tk * kCols + c1] = total[nt][i][2];
            wred[(tk + 1) * kCols + c1] = total[nt][i][3];
        }
    __syncthreads();
    for (uint32_t idx = threadIdx.x; idx < NT * 8 * kCols; idx += blockDim.x) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w * NT * 8 * kCols + idx];
        part[idx] = s;
    }

    auto store = [&](uint32_t tok, uint32_t c, float v) {
        if (tok < a.m && col0 + c < n) out[(size_t)tok * n + col0 + c] = v;
    };
    if (split == 1) {
        __syncthreads();
        for (uint32_t idx = threadIdx.x; idx < NT * 8 * kCols; idx += blockDim.x)
            store(idx / kCols, idx % kCols, part[idx]);
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const uint32_t c_lo = (kCols * blockIdx.y) / split, c_hi = (kCols * (blockIdx.y + 1)) / split;
    const uint32_t span = c_hi - c_lo;
    for (uint32_t idx = threadIdx.x; idx < span * NT * 8; idx += blockDim.x) {
        const uint32_t tok = idx / span, c = c_lo + idx % span;
        float s = 0.0f;
        for (uint32_t rk = 0; rk < split; ++rk) s += cluster.map_shared_rank(part, rk)[tok * kCols + c];
        store(tok, c, s);
    }
    cluster.sync();
}

template <int NT>
cudaError_t launch_nt(const Int4Args &a, uint32_t split, cudaStream_t s) {
    const size_t smem = (size_t)(kWarps + 1) * NT * 8 * kCols * sizeof(float);
    // opt in to more than 48 KB of dynamic shared memory once per device
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(int4_qkv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.tiles_q + 2 * a.tiles_kv, split, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, int4_qkv_kernel<NT>, a);
}

}  // namespace

// Split of K across a cluster: the smallest power of two (<= 8) that puts at
// least one CTA on every SM, while every warp keeps at least one group.
static uint32_t choose_split(const Int4Args &a) {
    const uint32_t tiles = a.tiles_q + 2 * a.tiles_kv;
    const uint32_t want = (uint32_t)device_sm_count();
    uint32_t split = 1;
    while (split < 8 && 2 * split * kWarps <= a.groups && tiles * split < want) split *= 2;
    return split;
}

cudaError_t launch_int4_qkv(const Int4Args &a, cudaStream_t s) {
    const uint32_t split = choose_split(a);
    return a.m <= 8 ? launch_nt<1>(a, split, s) : launch_nt<2>(a, split, s);
}

}  // namespace qdl
