// Internal declarations of libqdl: kernel argument blocks, launchers and
// small device helpers (inline PTX).  Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qdl.h"

namespace qdl {

#ifndef QDL_INT4_CC_MAX_ROWS
// token rows (at most 8) up to which the AWQ projection takes the CUDA-core
// stream-K kernel, also where the tcgen05 kernel applies.  Measured on the
// K=4096 QKV projection (CUDA cores vs tcgen05): 8.3 vs 12.0 us at M=1,
// 12.3 vs 12.2 us at M=4, 19.2 us at M=8 vs 13.6 us at M=16.
#define QDL_INT4_CC_MAX_ROWS 4
#endif
#ifndef QDL_INT4_TC_PASS_ROWS
// token rows per pass of the tcgen05 AWQ kernel (16 or 32).  Measured on the
// K=4096 QKV projection: one 32-row pass takes 28.3 us, one 16-row pass
// 13.2 us, so more rows go faster in passes of 16
#define QDL_INT4_TC_PASS_ROWS 16
#endif
#ifndef QDL_TUNE_EARLY_TRIGGER
// 1: the activation quantiser releases the GEMV before its own dependency
// wait, so consecutive calls overlap (the next GEMV streams weights while the
// previous one finishes)
#define QDL_TUNE_EARLY_TRIGGER 1
#endif
#ifndef QDL_TUNE_PDL
#define QDL_TUNE_PDL 1  // programmatic dependent launch between the library's kernels
#endif

constexpr int kMaxRows = QDL_MAX_ROWS;
constexpr int kKUnit = QDL_K_UNIT;

// ---------------------------------------------------------------- arguments

struct ActQuantArgs {
    const uint16_t *a;  // x, or gate for the SiLU variant (bf16 bits)
    const uint16_t *b;  // up for the SiLU variant, else unused
    uint32_t lda, ldb;  // row strides in elements
    uint32_t rows, k;
    uint8_t *q;         // [rows, k]
    float *s;           // [rows] or [rows, k/128]
    // optional: f32 output [rows, zn] (row stride zldc) to set to zero after
    // the dependency wait, for a following GEMV that accumulates into it
    float *zout;
    uint32_t zldc, zn;
};

struct W8A8Args {
    const uint8_t *q;   // activation codes [rows, k]
    const float *sa;    // activation scales [rows] or [rows, k/128]
    const uint8_t *w0, *w1, *w2;  // segment codes [n_s, k]
    const float *sw0, *sw1, *sw2; // segment scales
    void *out;
    uint32_t ldc;
    uint32_t out_bf16;
    uint32_t m;         // token rows in this launch
    uint32_t n, k;      // total output width, reduction length
    uint32_t n1, n2;    // segment split points
    uint32_t kb;        // k / 128
    uint32_t debug_skip_iter;  // self-test only: pipeline stage never loaded (else ~0u)
    uint64_t wait_limit_ns;    // limit of every device-side wait
    uint32_t accumulate;       // f32 output: out += y, split-K ranks add their partials atomically
    uint32_t out_zeroed;       // with accumulate: out was set to zero by the quantiser (a plain store suffices)
    uint32_t early_trigger;    // set by the launcher: release dependent kernels at the start
};

struct Int4Args {
    const float *x;     // [m, k]
    const uint32_t *qw0, *qw1, *qw2;
    const float *sc0, *sc1, *sc2;
    const float *zr0, *zr1, *zr2;
    float *out0, *out1, *out2;
    uint32_t m, k, group, groups;
    uint32_t nq, nkv;
    uint32_t tiles_q, tiles_kv;  // 128-column tiles per projection
    uint32_t vec2;               // 8-byte weight loads allowed
};

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.  Arguments are validated by
// the C-ABI layer before these are called.

struct PlanInfo {
    int kernel;
    uint32_t mma_n, tiles, split, stages, threads, smem;
    int clusters;
};
cudaError_t plan_w8a8_gemm_tc(const W8A8Args &a, int format, PlanInfo *p);

cudaError_t launch_act_quant(const ActQuantArgs &a, int format, bool silu, cudaStream_t s);
cudaError_t launch_w8a8_gemm_tc(const W8A8Args &a, int format, const uint8_t *const seg_w[3],
                                const uint32_t seg_n[3], cudaStream_t s);
cudaError_t read_and_clear_tc_fault(uint32_t *value);
uint32_t tc_bucket(uint32_t m);  // MMA N of the tensor-core kernel for m token rows
// true when the accumulating Block128 GEMV for these rows runs stream-K
// (one range of (tile, K block) units per CTA; the projection zeroes its f32
// output for it)
bool w8a8_streamk_applies(int format, uint32_t rows);
// Split-K factor minimising waves x (K blocks per CTA + fixed cost), where a
// split CTA also pays reduce_cost (in K-block units) for the cluster reduction;
// slots[s-1]: CTAs resident at once when launched in clusters of s.
uint32_t choose_split_k(uint32_t tiles, uint32_t kb, const uint32_t *slots, double reduce_cost);
void resident_cta_slots(const void *func, int threads, size_t smem, int per_sm, uint32_t *out);
cudaError_t launch_int4_qkv(const Int4Args &a, cudaStream_t s);
bool int4_tc_supported(uint32_t nq, uint32_t nkv, uint32_t group);
cudaError_t launch_int4_qkv_tc(const Int4Args &a, cudaStream_t s);  // up to QDL_INT4_TC_PASS_ROWS token rows
cudaError_t read_and_clear_int4_fault(uint32_t *value);
// zeroes the three f32 outputs [m, n_p] for a kernel that adds into them
cudaError_t launch_int4_zero(const Int4Args &a, cudaStream_t s);
bool int4_cc_supported(uint32_t nq, uint32_t nkv);                  // widths multiples of 32
cudaError_t launch_int4_qkv_cc(const Int4Args &a, cudaStream_t s);  // 1..8 token rows, CUDA cores
cudaError_t read_and_clear_int4cc_fault(uint32_t *value);

// KV-cache quantisers (kv_cache_quant.wgsl); arguments checked by the C ABI
cudaError_t launch_kv_quant_int8(const float *x, uint32_t tokens, uint32_t dim, int8_t *q, float *scale, cudaStream_t s);
cudaError_t launch_kv_dequant_int8(const int8_t *q, const float *scale, uint32_t tokens, uint32_t dim, float *out,
                                   cudaStream_t s);
cudaError_t launch_kv_quant_int4(const float *x, size_t n, uint32_t group, uint8_t *packed, float *scale, float *zero,
                                 cudaStream_t s);
cudaError_t launch_kv_dequant_int4(const uint8_t *packed, const float *scale, const float *zero, size_t n,
                                   uint32_t group, float *out, cudaStream_t s);

// weight preparation (FP8 per row / 128x128 block, AWQ packing); arguments
// checked by the C ABI
cudaError_t launch_fp8_weight_quant(int format, const void *w, bool bf16, uint32_t ldw, uint32_t n, uint32_t k,
                                    uint8_t *codes, float *scales, cudaStream_t s);
cudaError_t launch_awq_pack(const uint8_t *nib, uint32_t k, uint32_t n, uint32_t *qw, cudaStream_t s);

int device_sm_count();  // of the current device, cached

// ---------------------------------------------------------------- device helpers

#if defined(__CUDACC__)

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// Two binary32 values to two E4M3 codes, round to nearest even, saturating
// to +-448; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The library's exp in binary32: Cody and Waite reduction x = n ln2 + r,
// n = rint(x log2 e), ln2 split into RN32(ln2) and RN32(ln2 - RN32(ln2));
// e^r by the degree-7 Taylor polynomial (coefficients 1/j! rounded to
// binary32) in Horner form with fused multiply-adds; then an exact
// multiplication by 2^n (two steps when the result is subnormal).  Every
// operation is a correctly rounded binary32 operation, so the result is
// reproducible bit for bit.  Arguments above RN32(ln FLT_MAX) give +inf,
// below RN32(ln 2^-150) give +0.
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((n + 127) << 23); }

__device__ __forceinline__ float qdl_expf(float x) {
    if (x != x) return x;
    if (x > __uint_as_float(0x42b17218u)) return __int_as_float(0x7f800000);
    if (x < __uint_as_float(0xc2cff1b4u)) return 0.0f;
    const float t = __fmul_rn(x, __uint_as_float(0x3fb8aa3bu));
    const float n = rintf(t);
    float r = __fmaf_rn(-n, __uint_as_float(0x3f317218u), x);
    r = __fmaf_rn(-n, __uint_as_float(0xb102e308u), r);
    float p = __uint_as_float(0x39500d01u);          // 1/7!
    p = __fmaf_rn(p, r, __uint_as_float(0x3ab60b61u)); // 1/6!
    p = __fmaf_rn(p, r, __uint_as_float(0x3c088889u)); // 1/5!
    p = __fmaf_rn(p, r, __uint_as_float(0x3d2aaaabu)); // 1/4!
    p = __fmaf_rn(p, r, __uint_as_float(0x3e2aaaabu)); // 1/3!
    p = __fmaf_rn(p, r, 0.5f);                         // 1/2!
    p = __fmaf_rn(p, r, 1.0f);                         // 1/1!
    p = __fmaf_rn(p, r, 1.0f);                         // 1/0!
    int ni = static_cast<int>(n);
    if (ni > 127) {
        p = __fmul_rn(p, 2.0f);
        ni -= 1;
    }
    if (ni >= -126) return __fmul_rn(p, pow2i(ni));
    return __fmul_rn(__fmul_rn(p, pow2i(ni + 64)), pow2i(-64));
}

// SiLU(g) * u, one binary32 operation per step.
__device__ __forceinline__ float silu_mul(float g, float u) {
    const float e = qdl_expf(-g);
    const float d = __fadd_rn(1.0f, e);
    const float s = __fdiv_rn(g, d);
    return __fmul_rn(s, u);
}

// Loads of data that an earlier kernel on the stream writes (activations,
// activation scales, KV values and codes, weights being quantised).  The
// kernels are launched with programmatic stream serialisation, so they may
// start while that kernel still runs and read such data only after
// griddepcontrol.wait.  A non-coherent load (ld.global.nc, __ldg) is valid only
// for data that no kernel writes while this one runs, and the compiler may
// schedule it before the wait; these are plain coherent loads, in volatile asm
// so that they stay after the wait.
__device__ __forceinline__ float ld_dep(const float *p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_dep(const float4 *p) {
    float4 v;
    asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_dep(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint2 ld_dep(const uint2 *p) {
    uint2 v;
    asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_dep(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Streaming 16-byte load of data read exactly once (weights): bypass L1 and
// mark the lines evict-first in L2 so activations and scales stay resident.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t policy) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(policy));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void *p, uint64_t policy) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p), "l"(policy));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p, uint64_t policy) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                 : "=r"(r)
                 : "l"(p), "l"(policy));
    return r;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Read-only load through L1 (small operands shared by every warp of a CTA).
__device__ __forceinline__ uint4 ld_ro_v4(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

#endif  // __CUDACC__

}  // namespace qdl
