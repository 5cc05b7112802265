// W8A8 decode GEMV / skinny GEMM on the 5th-generation tensor cores
// (w8a8_decode.rs fn w8a8_gemv; segment routing from W8a8Weight::boundaries;
// scale layouts from enum W8a8Scale).  One pass over the weights for any
// token count up to 256.
//
//   y[m, j] = sum_kb Sa(m, kb) Sw(j, kb) sum_{k in kb} dec(q[m,k]) dec(W[j,k])
//
// Roles (one CTA = 128 output rows x a range of 128-wide K blocks):
//   warp 0, one lane : TMA producer.  Per K block, eight 16-row x 128-byte
//                      weight boxes (from the segment holding those rows) and
//                      one NTOK-row activation box land in a shared-memory
//                      stage (128-byte swizzle = the canonical K-major SW128
//                      operand layout), completing on the stage's mbarrier.
//   warp 1           : allocates the tensor memory; one lane issues
//                      tcgen05.mma kind::f8f6f4 (M = 128 weight rows,
//                      N = NTOK tokens, K = 32 per instruction, four per
//                      block) and commits each stage back to its `empty`
//                      mbarrier.
//   warps 2..        : epilogue, reading the f32 accumulators with tcgen05.ld.
//
// Scales.  PerRow: the accumulator sums the CTA's whole K range; the epilogue
// multiplies by sa[m] sw[j].  Block128: each 128-block accumulates into one of
// two TMEM buffers (ping-pong); the epilogue folds buffer b into register
// totals with sa[m, kb] sw[j/128, kb] while the tensor core fills the other.
//
// Split-K CTAs of one cluster reduce their partials through distributed shared
// memory in rank order (deterministic).  Every wait is bounded; after a
// timeout the CTA records a fault word, waits (bounded) for its copies and
// MMAs in flight, frees its tensor memory and returns.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <mutex>
#include <vector>

#include "tma_pipe.cuh"

namespace cg = cooperative_groups;

namespace qdl {

static __device__ uint32_t g_tc_fault;

namespace {

constexpr int kTileRows = 128;
constexpr uint32_t kWBytes = kTileRows * 128;  // weight tile per stage
constexpr uint32_t kWBox = 16 * 128;
#ifndef QDL_TC_STAGE_BYTES
#define QDL_TC_STAGE_BYTES (64 * 1024)
#endif
#ifndef QDL_TC_BIGBOX
#define QDL_TC_BIGBOX 1
#endif

constexpr uint32_t pow2_at_least(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

template <int NTOK, bool kBlock>
struct Tc {
    static constexpr uint32_t kABytes = NTOK * 128;
    static constexpr uint32_t kStage = kWBytes + kABytes;  // multiple of 1024 (NTOK % 8 == 0)
    // pipeline depth: as many stages as fit a per-CTA budget, at least 3
    static constexpr int kStages = (QDL_TC_STAGE_BYTES / kStage) < 3 ? 3 : (QDL_TC_STAGE_BYTES / kStage);
    static constexpr uint32_t kBarOff = kStages * kStage;
    static constexpr uint32_t kBytes = kBarOff + 256;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static constexpr int kEpi = kBlock ? (NTOK <= 64 ? 4 : NTOK / 16) : 4;  // epilogue warps
    static constexpr int kCpt = kBlock ? NTOK * 4 / kEpi : 16;               // columns per epilogue thread
    static constexpr int kThreads = (2 + kEpi) * 32;
    static constexpr uint32_t kTmemCols = pow2_at_least(kBlock ? 2 * NTOK : NTOK);
    static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(kTileRows * NTOK * 4 <= kBarOff, "reduction buffer must fit in the stage area");
    static_assert(kTmemCols <= 512, "tensor memory");
};

// ---------------------------------------------------------------- tcgen05 PTX

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (8-row x 128-byte atoms stacked at 1024-byte stride).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;                    // descriptor version
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B e4m3, both K-major.
template <int NTOK>
__device__ __forceinline__ constexpr uint32_t idesc_f8() {
    return (1u << 4) | ((uint32_t)(NTOK >> 3) << 17) | ((uint32_t)(kTileRows >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- kernel

template <int NTOK, bool kBlock>
__global__ void __launch_bounds__(Tc<NTOK, kBlock>::kThreads, 1)
    w8a8_gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                        const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                        const __grid_constant__ CUtensorMap tm_a, const W8A8Args a) {
    using C = Tc<NTOK, kBlock>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + C::kStages;
    uint64_t *accf = empty + C::kStages;  // [2] accumulator buffer ready
    uint64_t *acce = accf + 2;           // [2] accumulator buffer drained
    uint64_t *done = acce + 2;           // all MMAs complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    float *red = reinterpret_cast<float *>(smem);  // [NTOK][128], reuses the stages at the end

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tile_row0 = blockIdx.x * kTileRows;
    const uint32_t split = gridDim.y, sidx = blockIdx.y;
    const uint32_t kb0 = (a.kb * sidx) / split, kb1 = (a.kb * (sidx + 1)) / split;
    const uint32_t niter = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], C::kEpi);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fault = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(&g_tc_fault, code);
    };
    auto wait = [&](uint64_t *bar, uint32_t parity, uint32_t code) {
        if (!*abort_flag && !mbar_wait(bar, parity, a.wait_limit_ns)) fault(code);
    };

    // segment of this tile's first row (Block128 tiles never straddle segments)
    const float *tile_scale;
    const CUtensorMap *tile_big;
    uint32_t tile_lrow0, seg_end;
    if (tile_row0 < a.n1) {
        tile_scale = a.sw0; tile_lrow0 = tile_row0; tile_big = &tm_b0; seg_end = a.n1;
    } else if (tile_row0 < a.n2) {
        tile_scale = a.sw1; tile_lrow0 = tile_row0 - a.n1; tile_big = &tm_b1; seg_end = a.n2;
    } else {
        tile_scale = a.sw2; tile_lrow0 = tile_row0 - a.n2; tile_big = &tm_b2; seg_end = a.n;
    }
    // true when rows tile_row0 .. tile_row0+127 that exist all belong to that segment
    const bool tile_single = tile_row0 + kTileRows <= seg_end || seg_end == a.n;

    uint32_t issued = 0;
    constexpr int kCpt = C::kCpt;
    float total[kBlock ? kCpt : 1];
#pragma unroll
    for (int j = 0; j < (kBlock ? kCpt : 1); ++j) total[j] = 0.0f;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(tile_big);
            prefetch_tmap(&tm_a);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t slot = it % C::kStages, ph = (it / C::kStages) & 1;
                wait(&empty[slot], ph ^ 1, 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], C::kStage);
                issued = it + 1;
                if (it == a.debug_skip_iter) continue;  // self-test: this stage never lands
                uint8_t *st = smem + slot * C::kStage;
                const int32_t kk = (int32_t)((kb0 + it) * 128);
                if (QDL_TC_BIGBOX && tile_single) {
                    // the whole tile lies in one segment: one 128-row box
                    tma_load_2d(st, tile_big, kk, (int32_t)tile_lrow0, &full[slot], pol_w);
                } else {
#pragma unroll 1
                    for (int b = 0; b < kTileRows / 16; ++b) {
                        const uint32_t r0 = tile_row0 + 16 * b;
                        const CUtensorMap *m;
                        uint32_t lr;
                        if (r0 < a.n1) {
                            m = &tm_w0; lr = r0;
                        } else if (r0 < a.n2) {
                            m = &tm_w1; lr = r0 - a.n1;
                        } else {
                            m = &tm_w2; lr = r0 - a.n2;
                        }
                        tma_load_2d(st + b * kWBox, m, kk, (int32_t)lr, &full[slot], pol_w);
                    }
                }
                tma_load_2d(st + kWBytes, &tm_a, kk, 0, &full[slot], pol_a);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f8<NTOK>();
            const uint32_t sbase = smem_u32(smem);
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t slot = it % C::kStages, ph = (it / C::kStages) & 1;
                const uint32_t b = kBlock ? (it & 1) : 0;
                if (kBlock) wait(&acce[b], ((it >> 1) & 1) ^ 1, 4);
                wait(&full[slot], ph, 8);
                if (*abort_flag) break;
                tc_fence_after();
                const uint64_t ad = sw128_desc(sbase + slot * C::kStage);
                const uint64_t bd = sw128_desc(sbase + slot * C::kStage + kWBytes);
                const uint32_t d = tmem + b * NTOK;
#pragma unroll
                for (int k = 0; k < 4; ++k)  // K = 32 bytes per instruction: +2 in descriptor units
                    tc_mma(d, ad + 2 * k, bd + 2 * k, idesc, (kBlock ? k > 0 : (it > 0 || k > 0)) ? 1u : 0u);
                tc_commit(&empty[slot]);
                if (kBlock) tc_commit(&accf[b]);
            }
            tc_commit(done);  // completes once every MMA issued above has
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - 2;
        const int quad = warp & 3;                // TMEM lanes 32*quad .. 32*quad+31
        const int cgrp = e >> 2;                  // column group
        const uint32_t lrow = 32 * quad + lane;   // row within the tile
        const uint32_t row = tile_row0 + lrow;
        const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
        if constexpr (kBlock) {
            constexpr int kSRegs = (kCpt + 31) / 32;  // scale registers per lane
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t b = it & 1, kb = kb0 + it;
                // lane l holds sa[token cgrp*kCpt + 32r + l, kb] * sw; shuffled out below
                const float sw = tile_row0 < a.n ? __ldg(tile_scale + (size_t)(tile_lrow0 >> 7) * a.kb + kb) : 0.0f;
                float sreg[kSRegs];
#pragma unroll
                for (int r = 0; r < kSRegs; ++r) {
                    const uint32_t tok = cgrp * kCpt + 32 * r + lane;
                    sreg[r] = (32 * r + lane < (uint32_t)kCpt && tok < a.m) ? __ldg(a.sa + (size_t)tok * a.kb + kb) * sw
                                                                            : 0.0f;
                }
                wait(&accf[b], (it >> 1) & 1, 16);
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kCpt / 16; ++c) {
                    float v[16];
                    tc_ld16(taddr + b * NTOK + cgrp * kCpt + 16 * c, v);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int j = 16 * c + i;
                        const float s = __shfl_sync(0xffffffffu, sreg[j >> 5], j & 31);
                        total[j] = fmaf(v[i], s, total[j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce[b]);
            }
        } else {
            wait(done, 0, 32);
            tc_fence_after();
        }
    }

    // ---------------------------------------------------------------- drain after a timeout
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t first = issued > (uint32_t)C::kStages ? issued - C::kStages : 0;
            for (uint32_t it = first; it < issued; ++it)
                if (it != a.debug_skip_iter) mbar_wait(&full[it % C::kStages], (it / C::kStages) & 1, a.wait_limit_ns);
        }
        if (warp == 1 && lane == 0) mbar_wait(done, 0, a.wait_limit_ns);
        __syncthreads();
    }

    auto store = [&](uint32_t tok, uint32_t r, float v) {
        if (tok < a.m && r < a.n) {
            if (a.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)tok * a.ldc + r] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float *>(a.out)[(size_t)tok * a.ldc + r] = v;
        }
    };

    // ---------------------------------------------------------------- output
    // Each epilogue thread owns one row and a range of token columns; with
    // split > 1 it writes them to red[token][row] for the cluster reduction.
    if (warp >= 2) {
        const int e = warp - 2;
        const int quad = warp & 3;
        const int cgrp = e >> 2;
        const uint32_t lrow = 32 * quad + lane;
        const uint32_t row = tile_row0 + lrow;
        if constexpr (kBlock) {
#pragma unroll
            for (int j = 0; j < kCpt; ++j) {
                const uint32_t tok = cgrp * kCpt + j;
                if (split == 1)
                    store(tok, row, total[j]);
                else
                    red[tok * kTileRows + lrow] = total[j];
            }
        } else {
            // PerRow: scale the accumulator by sa[token] sw[row], 16 columns at a time
            const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
            uint32_t lr;
            const float *sseg;
            if (row < a.n1) {
                sseg = a.sw0; lr = row;
            } else if (row < a.n2) {
                sseg = a.sw1; lr = row - a.n1;
            } else {
                sseg = a.sw2; lr = row - a.n2;
            }
            const float swr = row < a.n ? __ldg(sseg + lr) : 0.0f;
            for (int c = 0; c < NTOK / 16; ++c) {  // every token column of this warp's 32 rows
                float v[16];
                tc_ld16(taddr + 16 * c, v);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t tok = 16 * c + i;
                    const float s = tok < a.m ? __ldg(a.sa + tok) * swr : 0.0f;
                    if (split == 1)
                        store(tok, row, v[i] * s);
                    else
                        red[tok * kTileRows + lrow] = v[i] * s;
                }
            }
            (void)e;
            (void)cgrp;
        }
    }

    if (split > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const uint32_t r_lo = (kTileRows * sidx) / split, r_hi = (kTileRows * (sidx + 1)) / split;
        const uint32_t span = r_hi - r_lo;
        const uint32_t m_used = a.m < (uint32_t)NTOK ? a.m : (uint32_t)NTOK;
        const float *peer[8];
#pragma unroll
        for (int rk = 0; rk < 8; ++rk) peer[rk] = cluster.map_shared_rank(red, rk < (int)split ? rk : 0);
        for (uint32_t idx = threadIdx.x; idx < span * m_used; idx += blockDim.x) {
            const uint32_t tok = idx / span, lr = r_lo + idx % span;
            float v[8];
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) v[rk] = rk < (int)split ? peer[rk][tok * kTileRows + lr] : 0.0f;
            float sum = 0.0f;
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) sum += v[rk];  // rank order; absent ranks add +0
            store(tok, tile_row0 + lr, sum);
        }
        cluster.sync();
    }

    // ---------------------------------------------------------------- free the tensor memory
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

template <int NTOK, bool kBlock>
int occupancy_tc() {
    using C = Tc<NTOK, kBlock>;
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        cudaFuncSetAttribute(w8a8_gemm_tc_kernel<NTOK, kBlock>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kAlloc);
        cache[dev] = resident_ctas((const void *)w8a8_gemm_tc_kernel<NTOK, kBlock>, C::kThreads, C::kAlloc,
                                   C::kTmemCols);
    }
    return cache[dev];
}

template <int NTOK, bool kBlock>
cudaError_t launch_tc_variant(const W8A8Args &a, const CUtensorMap (&maps)[7], cudaStream_t s) {
    using C = Tc<NTOK, kBlock>;
    const uint32_t tiles = (a.n + kTileRows - 1) / kTileRows;
    const uint32_t slots = (uint32_t)(device_sm_count() * occupancy_tc<NTOK, kBlock>());
    const uint32_t split = choose_split_k(tiles, a.kb, slots);
    (void)sizeof(C);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, split, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w8a8_gemm_tc_kernel<NTOK, kBlock>, maps[0], maps[1], maps[2], maps[3], maps[4],
                              maps[5], maps[6], a);
}

template <bool kBlock>
cudaError_t launch_tc_rows(const W8A8Args &a, const CUtensorMap (&maps)[7], uint32_t ntok, cudaStream_t s) {
    switch (ntok) {
        case 16: return launch_tc_variant<16, kBlock>(a, maps, s);
        case 32: return launch_tc_variant<32, kBlock>(a, maps, s);
        case 64: return launch_tc_variant<64, kBlock>(a, maps, s);
        case 128: return launch_tc_variant<128, kBlock>(a, maps, s);
        default: return launch_tc_variant<256, kBlock>(a, maps, s);
    }
}

}  // namespace

// Token-count bucket of the tensor-core kernel: the MMA's N (16..256).
uint32_t tc_bucket(uint32_t m) {
    uint32_t n = 16;
    while (n < m) n <<= 1;
    return n;
}

cudaError_t launch_w8a8_gemm_tc(const W8A8Args &a, int format, const uint8_t *const seg_w[3], const uint32_t seg_n[3],
                                cudaStream_t s) {
    CUtensorMap maps[7];  // 16-row boxes x3, 128-row boxes x3, activations
    for (int i = 0; i < 3; ++i) {
        cudaError_t e = make_tmap_u8(&maps[i], seg_w[i], a.k, seg_n[i], a.k, 128, 16);
        if (e != cudaSuccess) return e;
        e = make_tmap_u8(&maps[3 + i], seg_w[i], a.k, seg_n[i], a.k, 128, kTileRows);
        if (e != cudaSuccess) return e;
    }
    const uint32_t ntok = tc_bucket(a.m);
    cudaError_t e = make_tmap_u8(&maps[6], a.q, a.k, a.m, a.k, 128, ntok);
    if (e != cudaSuccess) return e;
    return format == QDL_SCALE_BLOCK128 ? launch_tc_rows<true>(a, maps, ntok, s) : launch_tc_rows<false>(a, maps, ntok, s);
}

cudaError_t read_and_clear_tc_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_tc_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_tc_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
