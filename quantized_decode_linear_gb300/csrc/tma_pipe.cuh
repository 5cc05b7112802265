// TMA tensor maps, mbarrier pipelines and bounded waits (inline PTX for
// sm_103a).  Shared by the kernels that stream weight tiles through shared
// memory.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "qdl_internal.cuh"

namespace qdl {

// Host: 2D row-major u8 tensor [rows, cols] with row stride `stride` bytes,
// copied in boxes of box_cols bytes x box_rows rows with the 128-byte
// swizzle (box_cols must be 128).  Returns cudaSuccess or an error.
cudaError_t make_tmap_u8(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t stride,
                         uint32_t box_cols, uint32_t box_rows);
// packed AWQ words [rows, words] u32, box 32 words x box_rows rows, 128-byte swizzle
cudaError_t make_tmap_words(CUtensorMap *map, const void *base, uint64_t words, uint64_t rows, uint32_t box_rows);
// x [rows, k] f32, box 32 values x box_rows rows, 128-byte swizzle; rows past the end read as zero
cudaError_t make_tmap_f32(CUtensorMap *map, const float *x, uint64_t k, uint64_t rows, uint32_t box_rows);

// [outer, inner] row-major tensor of 4-byte elements of `type`, row pitch
// inner * 4 bytes, box box_inner x box_outer, the given swizzle; elements past
// either end read as zero
cudaError_t make_tmap_4b(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
// [outer, inner] row-major tensor of 4-byte elements (u32 codes, or f32 when
// `f32`), row pitch inner * 4 bytes, box box_inner x box_outer, no swizzle;
// elements past either end read as zero
cudaError_t make_tmap_plain(CUtensorMap *map, bool f32, const void *base, uint64_t inner, uint64_t outer,
                            uint32_t box_inner, uint32_t box_outer);

// CTAs of a kernel that can be resident on one SM at once.
int resident_ctas(const void *func, int threads, size_t smem, int tmem_cols);

// Default limit of every bounded device-side wait.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make initialised barriers visible to the async (TMA) proxy and the cluster
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with parity `parity` to complete, giving up
// after limit_ns nanoseconds.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-byte asynchronous copy global -> shared (through L1: a coherent read, so
// valid for data an earlier kernel wrote once the dependency wait returned),
// and the per-thread groups that track completion.
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's committed groups are still pending
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 2D tiled TMA load into this CTA's shared memory, completing on `bar`.
// c0 is the innermost (byte) coordinate and must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t c0, int32_t c1, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// generic-proxy shared-memory writes -> visible to the async proxy (TMA,
// tensor core)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

#endif  // __CUDACC__

}  // namespace qdl
