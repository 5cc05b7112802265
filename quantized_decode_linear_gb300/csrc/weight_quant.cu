// Weight preparation on the GPU: FP8 E4M3 weight quantisation per output row
// or per 128x128 block, and AWQ packing of 4-bit codes.
//
// FP8 (the weight side of the scale layouts of w8a8_decode.rs, enum
// W8a8Scale; scale absmax / 448 as the workloads state for weights):
//   s    = absmax over the row / block / 448     (binary32 division)
//   code = e4m3(w / s)                           (binary32 division, RNE, saturating)
// a row or block whose absmax is 0 gets s = 0 and the codes of its signed
// zeros.  One CTA of 512 threads per row or block: each thread keeps up to
// kChunks chunks of 8 values in registers between the absmax pass and the
// encode pass (128x128 blocks and rows up to 16384 values are read from
// memory once), the absmax is reduced across the CTA, and codes leave as
// 8-byte stores.  Small register footprint, so that several CTAs share an SM
// and the divisions of one overlap the loads of another.
//
// AWQ (fused_int4_qkv.rs, QKV_AWQ_SHIFTS; the inverse of unpack_awq_qkv):
// word j of row k holds the code of column 8j + i at bits SHIFT[i] ..
// SHIFT[i] + 3, SHIFT = {0, 16, 4, 20, 8, 24, 12, 28}.  One thread per
// packed word: an 8-byte load of 8 codes (low nibble of each byte), one
// 4-byte store.
#include "qdl_internal.cuh"

namespace qdl {

namespace {

constexpr int kThreadsW = 512;
constexpr int kChunks = 4;  // 8-value chunks a thread keeps in registers

template <bool kBf16>
__device__ __forceinline__ void load8(const void *base, size_t elem, float (&v)[8]) {
    if (kBf16) {
        const uint4 r = ld_dep(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + elem));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
            v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + elem);
        const float4 a = ld_dep(p), b = ld_dep(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ float wq_operand(float v, float s) { return s == 0.0f ? v : __fdiv_rn(v, s); }

// kBlock: region = 128x128 block (blockIdx.x = block row * kb + block col),
// else one row (blockIdx.x = row).  ldw in elements; k % 128 == 0.
template <bool kBf16, bool kBlock>
__global__ void __launch_bounds__(kThreadsW, 2) fp8_weight_quant_kernel(const void *w, uint32_t ldw, uint32_t n,
                                                                     uint32_t k, uint8_t *codes, float *scales) {
    __shared__ float warp_max[kThreadsW / 32];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // w may come from the previous kernel
    const uint32_t kb = k / 128;
    uint32_t r0, c0, rows, cpr;  // region origin, rows, 8-value chunks per region row
    if (kBlock) {
        const uint32_t br = blockIdx.x / kb, bc = blockIdx.x % kb;
        r0 = br * 128;
        c0 = bc * 128;
        rows = n - r0 < 128 ? n - r0 : 128;
        cpr = 16;
    } else {
        r0 = blockIdx.x;
        c0 = 0;
        rows = 1;
        cpr = k / 8;
    }
    const uint32_t nchunk = rows * cpr;
    auto elem_of = [&](uint32_t c) -> size_t {
        const uint32_t r = c / cpr, cc = c % cpr;
        return (size_t)(r0 + r) * ldw + c0 + 8 * cc;
    };
    auto out_of = [&](uint32_t c) -> size_t {
        const uint32_t r = c / cpr, cc = c % cpr;
        return (size_t)(r0 + r) * k + c0 + 8 * cc;
    };

    float keep[kChunks][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const uint32_t c = threadIdx.x + i * kThreadsW;
        if (c < nchunk) {
            load8<kBf16>(w, elem_of(c), keep[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(keep[i][e]));
        }
    }
    for (uint32_t c = threadIdx.x + kChunks * kThreadsW; c < nchunk; c += kThreadsW) {
        float v[8];
        load8<kBf16>(w, elem_of(c), v);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < kThreadsW / 32; ++i) amax = fmaxf(amax, warp_max[i]);
    const float s = __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) scales[blockIdx.x] = s;

    auto encode = [&](const float (&v)[8], uint32_t c) {
        uint2 q;
        q.x = cvt_e4m3x2(wq_operand(v[0], s), wq_operand(v[1], s)) |
              (cvt_e4m3x2(wq_operand(v[2], s), wq_operand(v[3], s)) << 16);
        q.y = cvt_e4m3x2(wq_operand(v[4], s), wq_operand(v[5], s)) |
              (cvt_e4m3x2(wq_operand(v[6], s), wq_operand(v[7], s)) << 16);
        *reinterpret_cast<uint2 *>(codes + out_of(c)) = q;
    };
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const uint32_t c = threadIdx.x + i * kThreadsW;
        if (c < nchunk) encode(keep[i], c);
    }
    for (uint32_t c = threadIdx.x + kChunks * kThreadsW; c < nchunk; c += kThreadsW) {
        float v[8];
        load8<kBf16>(w, elem_of(c), v);
        encode(v, c);
    }
    // no early release of dependents: the decode kernels stream weights
    // before their own dependency wait, so a kernel that writes weights must
    // have finished before the next one starts
}

__global__ void __launch_bounds__(256) awq_pack_kernel(const uint8_t *nib, uint32_t k, uint32_t n, uint32_t *qw) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t words = n / 8;
    const size_t total = (size_t)k * words;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += stride) {
        // word i = row i / words, word i % words: bytes 8 i .. 8 i + 7 of nib
        const uint2 b = ld_dep(reinterpret_cast<const uint2 *>(nib + 8 * i));
        constexpr int kShift[8] = {0, 16, 4, 20, 8, 24, 12, 28};
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t byte = ((j < 4 ? b.x : b.y) >> (8 * (j & 3))) & 0xFu;
            word |= byte << kShift[j];
        }
        qw[i] = word;
    }
    // no early release of dependents (see fp8_weight_quant_kernel)
}

cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

}  // namespace

cudaError_t launch_fp8_weight_quant(int format, const void *w, bool bf16, uint32_t ldw, uint32_t n, uint32_t k,
                                    uint8_t *codes, float *scales, cudaStream_t s) {
    const bool block = format == QDL_SCALE_BLOCK128;
    const uint64_t ctas = block ? (uint64_t)((n + 127) / 128) * (k / 128) : n;
    if (ctas == 0 || ctas > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kThreadsW, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    if (bf16)
        return block ? cudaLaunchKernelEx(&cfg, fp8_weight_quant_kernel<true, true>, w, ldw, n, k, codes, scales)
                     : cudaLaunchKernelEx(&cfg, fp8_weight_quant_kernel<true, false>, w, ldw, n, k, codes, scales);
    return block ? cudaLaunchKernelEx(&cfg, fp8_weight_quant_kernel<false, true>, w, ldw, n, k, codes, scales)
                 : cudaLaunchKernelEx(&cfg, fp8_weight_quant_kernel<false, false>, w, ldw, n, k, codes, scales);
}

cudaError_t launch_awq_pack(const uint8_t *nib, uint32_t k, uint32_t n, uint32_t *qw, cudaStream_t s) {
    const uint64_t words = (uint64_t)k * (n / 8);
    uint64_t ctas = (words + 255) / 256;
    const uint64_t cap = (uint64_t)device_sm_count() * 8;
    if (ctas > cap) ctas = cap;
    if (ctas == 0) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, awq_pack_kernel, nib, k, n, qw);
}

}  // namespace qdl
