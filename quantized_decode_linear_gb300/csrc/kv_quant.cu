// KV-cache quantisers and dequantisers (kv_cache_quant.wgsl:
// quantize_kv_fp8_per_token_f32, quantize_kv_int8_f32, quantize_kv_int4_f32,
// and the matching dequantize_* kernels).
//
// Per-token symmetric int8 (the page's "FP8" per-token kernel computes the
// same thing as its INT8 one: it scales to 127 and rounds to integers):
//   s = max(absmax / 127, 1e-8),  q = clamp(rint(v / s), -128, 127),  v' = q s
// Per-group asymmetric INT4 over the flattened [tokens, head_dim] array:
//   scale = (max - min) / 15,  zero = -min / max(scale, 1e-8),
//   q = clamp(rint((v - min) / max(scale, 1e-8)), 0, 15),
//   v' = q scale - zero scale
// with two codes per byte (even element in the low nibble).  rint rounds
// halves to even, as WGSL round() does.  Every step is one correctly rounded
// binary32 operation (__fdiv_rn, __fsub_rn, __fmul_rn: no contraction), so
// codes, scales and dequantised values are reproducible bit for bit.
//
// The kernels stream HBM: each warp issues all of its loads before the
// arithmetic, codes leave as 32-bit words, values as float4.
#include <stdint.h>

#include <type_traits>

#include "qdl_internal.cuh"

namespace qdl {

namespace {

constexpr int kKvThreads = 256;
constexpr int kKvWarps = kKvThreads / 32;
#ifndef QDL_KV_TOKENS_PER_WARP
#define QDL_KV_TOKENS_PER_WARP 2
#endif
#ifndef QDL_KV_ROUNDS
#define QDL_KV_ROUNDS 1
#endif
constexpr int kTokensPerWarp = QDL_KV_TOKENS_PER_WARP;  // int8 quantiser: tokens whose loads one warp keeps in flight

// Programmatic launch: release the next kernel at once, then wait for the
// previous one (the input may come from it, and it may still read the
// buffers written here).
__device__ __forceinline__ void kv_dependency_prologue() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float kv_scale_int8(float absmax) {
    const float s = __fdiv_rn(absmax, 127.0f);
    return s > 1e-8f ? s : 1e-8f;
}

__device__ __forceinline__ uint32_t q_int8(float v, float s) {
    float r = rintf(__fdiv_rn(v, s));
    r = fminf(fmaxf(r, -128.0f), 127.0f);
    return (uint32_t)(int32_t)r & 0xFFu;
}

// CH float4 chunks of a token per lane (head_dim <= 128 * CH, head_dim % 4 == 0)
template <int CH>
__global__ void __launch_bounds__(kKvThreads) kv_quant_int8_kernel(const float *__restrict__ x, uint32_t tokens,
                                                                    uint32_t dim, uint32_t *__restrict__ q,
                                                                    float *__restrict__ scale) {
    kv_dependency_prologue();
    const uint32_t warp = (blockIdx.x * kKvWarps + (threadIdx.x >> 5)), lane = threadIdx.x & 31;
    const uint32_t t0 = warp * kTokensPerWarp;
    const uint32_t chunks = dim / 4;
    float4 v[kTokensPerWarp][CH];
#pragma unroll
    for (int i = 0; i < kTokensPerWarp; ++i)
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const uint32_t t = t0 + i, ch = lane + 32 * c;
            v[i][c] = (t < tokens && ch < chunks) ? ld_dep(reinterpret_cast<const float4 *>(x + (size_t)t * dim) + ch)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
    for (int i = 0; i < kTokensPerWarp; ++i) {
        const uint32_t t = t0 + i;
        float m = 0.0f;
#pragma unroll
        for (int c = 0; c < CH; ++c)
            m = fmaxf(fmaxf(fmaxf(m, fabsf(v[i][c].x)), fmaxf(fabsf(v[i][c].y), fabsf(v[i][c].z))), fabsf(v[i][c].w));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float s = kv_scale_int8(m);
        if (t >= tokens) continue;  // whole warp
        if (lane == 0) scale[t] = s;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const uint32_t ch = lane + 32 * c;
            if (ch < chunks)
                q[(size_t)t * chunks + ch] = q_int8(v[i][c].x, s) | (q_int8(v[i][c].y, s) << 8) |
                                             (q_int8(v[i][c].z, s) << 16) | (q_int8(v[i][c].w, s) << 24);
        }
    }
}

// any head_dim % 4 == 0: one warp per token, two passes (the second from L1/L2)
__global__ void __launch_bounds__(kKvThreads) kv_quant_int8_wide_kernel(const float *__restrict__ x, uint32_t tokens,
                                                                         uint32_t dim, uint32_t *__restrict__ q,
                                                                         float *__restrict__ scale) {
    kv_dependency_prologue();
    const uint32_t t = blockIdx.x * kKvWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= tokens) return;
    const uint32_t chunks = dim / 4;
    const float4 *row = reinterpret_cast<const float4 *>(x + (size_t)t * dim);
    float m = 0.0f;
    for (uint32_t ch = lane; ch < chunks; ch += 32) {
        const float4 v = ld_dep(row + ch);
        m = fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = kv_scale_int8(m);
    if (lane == 0) scale[t] = s;
    for (uint32_t ch = lane; ch < chunks; ch += 32) {
        const float4 v = ld_dep(row + ch);
        q[(size_t)t * chunks + ch] = q_int8(v.x, s) | (q_int8(v.y, s) << 8) | (q_int8(v.z, s) << 16) | (q_int8(v.w, s) << 24);
    }
}

// v' = q s, four values (one code word) per thread and step
__global__ void __launch_bounds__(kKvThreads) kv_dequant_int8_kernel(const uint32_t *__restrict__ q,
                                                                      const float *__restrict__ scale, uint32_t tokens,
                                                                      uint32_t dim, float4 *__restrict__ out) {
    kv_dependency_prologue();
    const size_t words = (size_t)tokens * dim / 4;
    const uint32_t wpt = dim / 4;  // words per token
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride) {
        const uint32_t w = ld_dep(q + i);
        const float s = ld_dep(scale + i / wpt);
        float4 o;
        o.x = __fmul_rn((float)(int8_t)(w & 0xFF), s);
        o.y = __fmul_rn((float)(int8_t)((w >> 8) & 0xFF), s);
        o.z = __fmul_rn((float)(int8_t)((w >> 16) & 0xFF), s);
        o.w = __fmul_rn((float)(int8_t)(w >> 24), s);
        out[i] = o;
    }
}

struct Int4Fold {
    float mn, den, scale, zero;
};

__device__ __forceinline__ Int4Fold kv_fold_int4(float mn, float mx) {
    Int4Fold f;
    f.mn = mn;
    f.scale = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    f.den = f.scale > 1e-8f ? f.scale : 1e-8f;
    f.zero = __fdiv_rn(-mn, f.den);
    return f;
}

__device__ __forceinline__ uint32_t q_int4(float v, const Int4Fold &f) {
    float r = rintf(__fdiv_rn(__fsub_rn(v, f.mn), f.den));
    r = fminf(fmaxf(r, 0.0f), 15.0f);
    return (uint32_t)r;
}

// 8 values -> one word of 8 codes (value i in nibble i: even elements low)
__device__ __forceinline__ uint32_t pack_int4(const float4 &a, const float4 &b, const Int4Fold &f) {
    return q_int4(a.x, f) | (q_int4(a.y, f) << 4) | (q_int4(a.z, f) << 8) | (q_int4(a.w, f) << 12) |
           (q_int4(b.x, f) << 16) | (q_int4(b.y, f) << 20) | (q_int4(b.z, f) << 24) | (q_int4(b.w, f) << 28);
}

__device__ __forceinline__ void minmax8(const float4 &a, const float4 &b, float &mn, float &mx) {
    mn = fminf(fminf(fminf(a.x, a.y), fminf(a.z, a.w)), fminf(fminf(b.x, b.y), fminf(b.z, b.w)));
    mx = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
}

// group = 8 L with L a power of two <= 32: L lanes per group, one 8-value
// chunk per lane, 32 / L groups per warp and kRounds batches per warp with
// every load issued first
constexpr int kRounds = QDL_KV_ROUNDS;

template <int L>
__global__ void __launch_bounds__(kKvThreads) kv_quant_int4_kernel(const float *__restrict__ x, uint32_t groups,
                                                                    uint32_t *__restrict__ packed,
                                                                    float *__restrict__ scale, float *__restrict__ zero) {
    kv_dependency_prologue();
    constexpr uint32_t kGpw = 32 / L, kGroup = 8 * L;
    const uint32_t warp = blockIdx.x * kKvWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const uint32_t chunk = lane % L;
    float4 v[kRounds][2];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const uint32_t g = (warp * kRounds + r) * kGpw + lane / L;
        const float4 *p = reinterpret_cast<const float4 *>(x + (size_t)g * kGroup + 8 * chunk);
        const bool ok = g < groups;
        v[r][0] = ok ? ld_dep(p) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[r][1] = ok ? ld_dep(p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
        const uint32_t g = (warp * kRounds + r) * kGpw + lane / L;
        float mn, mx;
        minmax8(v[r][0], v[r][1], mn, mx);
#pragma unroll
        for (int o = L / 2; o > 0; o >>= 1) {  // within aligned runs of L lanes
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (g >= groups) continue;
        const Int4Fold f = kv_fold_int4(mn, mx);
        packed[((size_t)g * kGroup + 8 * chunk) / 8] = pack_int4(v[r][0], v[r][1], f);
        if (chunk == 0) {
            scale[g] = f.scale;
            zero[g] = f.zero;
        }
    }
}

// any group % 8 == 0: one warp per group, two passes (the second from L1/L2)
__global__ void __launch_bounds__(kKvThreads) kv_quant_int4_wide_kernel(const float *__restrict__ x, uint32_t groups,
                                                                         uint32_t group, uint32_t *__restrict__ packed,
                                                                         float *__restrict__ scale,
                                                                         float *__restrict__ zero) {
    kv_dependency_prologue();
    const uint32_t g = blockIdx.x * kKvWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (g >= groups) return;
    const uint32_t chunks = group / 8;
    const float4 *p = reinterpret_cast<const float4 *>(x + (size_t)g * group);
    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
    for (uint32_t c = lane; c < chunks; c += 32) {
        float a, b;
        minmax8(ld_dep(p + 2 * c), ld_dep(p + 2 * c + 1), a, b);
        mn = fminf(mn, a);
        mx = fmaxf(mx, b);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const Int4Fold f = kv_fold_int4(mn, mx);
    if (lane == 0) {
        scale[g] = f.scale;
        zero[g] = f.zero;
    }
    for (uint32_t c = lane; c < chunks; c += 32)
        packed[(size_t)g * chunks + c] = pack_int4(ld_dep(p + 2 * c), ld_dep(p + 2 * c + 1), f);
}

// v' = q scale - zero scale, eight values (one code word) per thread and step
__global__ void __launch_bounds__(kKvThreads) kv_dequant_int4_kernel(const uint32_t *__restrict__ packed,
                                                                      const float *__restrict__ scale,
                                                                      const float *__restrict__ zero, size_t words,
                                                                      uint32_t group, float4 *__restrict__ out) {
    kv_dependency_prologue();
    const uint32_t wpg = group / 8;  // words per group
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride) {
        const uint32_t w = ld_dep(packed + i);
        const size_t g = i / wpg;
        const float s = ld_dep(scale + g), zs = __fmul_rn(ld_dep(zero + g), s);
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = __fsub_rn(__fmul_rn((float)((w >> (4 * j)) & 0xFu), s), zs);
        out[2 * i] = make_float4(o[0], o[1], o[2], o[3]);
        out[2 * i + 1] = make_float4(o[4], o[5], o[6], o[7]);
    }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kv(void (*kernel)(KArgs...), uint32_t grid, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kKvThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

uint32_t grid_for(size_t work_items, uint32_t per_block) {
    const size_t b = (work_items + per_block - 1) / per_block;
    return (uint32_t)(b < 1 ? 1 : b);
}

// elementwise kernels: enough blocks to cover the SMs several times, then a grid-stride loop
uint32_t stream_grid(size_t items) {
    const size_t want = (items + kKvThreads - 1) / kKvThreads;
    const size_t cap = (size_t)device_sm_count() * 16;
    return (uint32_t)(want < 1 ? 1 : want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_kv_quant_int8(const float *x, uint32_t tokens, uint32_t dim, int8_t *q, float *scale, cudaStream_t s) {
    uint32_t *qw = reinterpret_cast<uint32_t *>(q);
    const uint32_t grid = grid_for(tokens, kKvWarps * kTokensPerWarp);
    if (dim <= 128) return launch_kv(kv_quant_int8_kernel<1>, grid, s, x, tokens, dim, qw, scale);
    if (dim <= 256) return launch_kv(kv_quant_int8_kernel<2>, grid, s, x, tokens, dim, qw, scale);
    if (dim <= 512) return launch_kv(kv_quant_int8_kernel<4>, grid, s, x, tokens, dim, qw, scale);
    return launch_kv(kv_quant_int8_wide_kernel, grid_for(tokens, kKvWarps), s, x, tokens, dim, qw, scale);
}

cudaError_t launch_kv_dequant_int8(const int8_t *q, const float *scale, uint32_t tokens, uint32_t dim, float *out,
                                   cudaStream_t s) {
    const size_t words = (size_t)tokens * dim / 4;
    return launch_kv(kv_dequant_int8_kernel, stream_grid(words), s, reinterpret_cast<const uint32_t *>(q), scale,
                     tokens, dim, reinterpret_cast<float4 *>(out));
}

cudaError_t launch_kv_quant_int4(const float *x, size_t n, uint32_t group, uint8_t *packed, float *scale, float *zero,
                                 cudaStream_t s) {
    const uint32_t groups = (uint32_t)(n / group);
    uint32_t *pw = reinterpret_cast<uint32_t *>(packed);
    auto launch = [&](auto tag) {
        constexpr int L = decltype(tag)::value;
        return launch_kv(kv_quant_int4_kernel<L>, grid_for(groups, kKvWarps * kRounds * (32 / L)), s, x, groups, pw,
                         scale, zero);
    };
    switch (group / 8) {  // lanes per group
        case 1: return launch(std::integral_constant<int, 1>());
        case 2: return launch(std::integral_constant<int, 2>());
        case 4: return launch(std::integral_constant<int, 4>());
        case 8: return launch(std::integral_constant<int, 8>());
        case 16: return launch(std::integral_constant<int, 16>());
        case 32: return launch(std::integral_constant<int, 32>());
        default: return launch_kv(kv_quant_int4_wide_kernel, grid_for(groups, kKvWarps), s, x, groups, group, pw, scale, zero);
    }
}

cudaError_t launch_kv_dequant_int4(const uint8_t *packed, const float *scale, const float *zero, size_t n,
                                   uint32_t group, float *out, cudaStream_t s) {
    const size_t words = n / 8;
    return launch_kv(kv_dequant_int4_kernel, stream_grid(words), s, reinterpret_cast<const uint32_t *>(packed), scale,
                     zero, words, group, reinterpret_cast<float4 *>(out));
}

}  // namespace qdl
