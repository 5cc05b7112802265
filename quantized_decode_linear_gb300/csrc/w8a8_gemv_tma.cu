// W8A8 decode GEMV for up to 16 token rows per launch (w8a8_decode.rs fn
// w8a8_gemv; segment routing from W8a8Weight::boundaries; scale layouts from
// enum W8a8Scale).  HBM-bound: every weight byte is read exactly once.
//
//   y[m, j] = sum_kb Sa(m, kb) Sw(j, kb) sum_{k in kb} dec(q[m,k]) dec(W[j,k])
//
// Pipeline.  A CTA owns 128 consecutive output rows and a range of 128-wide K
// blocks.  One producer lane streams, per K block, eight 16-row x 128-byte
// weight boxes (each from the segment that holds those rows) and one
// activation box (the token rows) into a shared-memory stage with 2D TMA
// copies (128-byte swizzle, evict-first for weights), completing on the
// stage's `full` mbarrier.  Eight consumer warps, one per 16-row box, wait on
// `full`, read their MMA fragments from shared memory and release the stage
// through its `empty` mbarrier.  STAGES stages are in flight per CTA.
//
// MMA.  m16n8k32 e4m3 x e4m3 -> f32 with the weights as the 16-row A
// operand and the tokens as the 8-column B operand.  Lane (g = lane/4,
// t = lane%4) reads 16 bytes of its rows at chunk 4c+t of the 128-byte row;
// the MMA's K index is permuted identically for A and B, which leaves the dot
// product unchanged.  A-row g is weight row P(g) and B-column n is token
// P(n), P = (0,4,1,5,2,6,3,7): with the swizzle, the eight lanes of every
// quarter warp then hit eight different 16-byte bank groups.
//
// Scales.  The MMA accumulates one 128-block; the block's partial sums are
// folded into f32 totals (Block128: times sa[m,kb] sw[j/128,kb]; PerRow: plain
// sum, scaled once at the end).  Split-K CTAs of one cluster reduce their
// partials through distributed shared memory in rank order (deterministic).
//
// Every mbarrier wait is bounded (a wait limit in nanoseconds); on timeout
// the CTA records a fault word that the host reads with
// qdl_check_device_fault, skips the remaining waits, drains its copies with
// bounded waits and still reaches every cluster barrier.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <mutex>
#include <vector>

#include "tma_pipe.cuh"

namespace cg = cooperative_groups;

#ifndef QDL_TUNE_STAGES
#define QDL_TUNE_STAGES 4
#endif

namespace qdl {

static __device__ uint32_t g_gemv_fault;

namespace {

constexpr int kConsumers = 8;                 // consumer warps, 16 rows each
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kRowsPerCta = kConsumers * 16;  // 128
constexpr int kStages = QDL_TUNE_STAGES;
constexpr uint32_t kWBox = 16 * 128;          // one 16-row weight box
constexpr uint32_t kWBytes = kConsumers * kWBox;

template <int NT>
struct Layout {
    static constexpr uint32_t kActRows = NT * 8;
    static constexpr uint32_t kABytes = kActRows * 128;
    static constexpr uint32_t kStage = kWBytes + kABytes;  // a multiple of 1024
    static constexpr uint32_t kBarOff = kStages * kStage;
    static constexpr uint32_t kRedOff = kBarOff + 2 * kStages * 8 + 16;
    static constexpr uint32_t kBytes = kRedOff + kActRows * kRowsPerCta * 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ int perm8(int g) { return (g >> 1) | ((g & 1) << 2); }

__device__ __forceinline__ void route(const W8A8Args &a, uint32_t row0, const CUtensorMap *m0, const CUtensorMap *m1,
                                      const CUtensorMap *m2, const CUtensorMap *&map, const float *&scale,
                                      uint32_t &lrow0) {
    if (row0 < a.n1) {
        map = m0; scale = a.sw0; lrow0 = row0;
    } else if (row0 < a.n2) {
        map = m1; scale = a.sw1; lrow0 = row0 - a.n1;
    } else {
        map = m2; scale = a.sw2; lrow0 = row0 - a.n2;
    }
}

template <int NT, bool kBlock>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_gemv_tma_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                         const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_a,
                         const W8A8Args a) {
    using L = Layout<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *empty = full + kStages;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(empty + kStages);
    float *red = reinterpret_cast<float *>(smem + L::kRedOff);  // [kActRows][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tile_row0 = blockIdx.x * kRowsPerCta;
    const uint32_t split = gridDim.y, sidx = blockIdx.y;
    const uint32_t kb0 = (a.kb * sidx) / split, kb1 = (a.kb * (sidx + 1)) / split;
    const uint32_t niter = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    auto fault = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(&g_gemv_fault, code);
    };

    float total[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) total[nt][j] = 0.0f;

    const CUtensorMap *wmap;
    const float *sseg;
    uint32_t lrow0 = 0;
    uint32_t issued = 0;  // stages the producer armed (producer lane only)

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_w0);
            prefetch_tmap(&tm_a);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t slot = it % kStages, ph = (it / kStages) & 1;
                if (!*abort_flag && !mbar_wait(&empty[slot], ph ^ 1, a.wait_limit_ns)) fault(1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], L::kStage);
                issued = it + 1;
                if (it == a.debug_skip_iter) continue;  // self-test: this stage never lands
                uint8_t *st = smem + slot * L::kStage;
                const int32_t kk = (int32_t)((kb0 + it) * 128);
#pragma unroll 1
                for (int b = 0; b < kConsumers; ++b) {
                    const CUtensorMap *m;
                    const float *unused;
                    uint32_t lr;
                    route(a, tile_row0 + 16 * b, &tm_w0, &tm_w1, &tm_w2, m, unused, lr);
                    tma_load_2d(st + b * kWBox, m, kk, (int32_t)lr, &full[slot], pol_w);
                }
                tma_load_2d(st + kWBytes, &tm_a, kk, 0, &full[slot], pol_a);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int g = lane >> 2, t = lane & 3;
        const int pg = perm8(g);
        const uint32_t row0 = tile_row0 + 16 * warp;
        route(a, row0, &tm_w0, &tm_w1, &tm_w2, wmap, sseg, lrow0);
        const bool warp_ok = row0 < a.n;
        const uint32_t smem_base = smem_u32(smem);
        for (uint32_t it = 0; it < niter; ++it) {
            const uint32_t slot = it % kStages, ph = (it / kStages) & 1;
            const uint32_t kb = kb0 + it;
            // block scales for this K block (loaded before the wait so that
            // their latency overlaps it)
            float s_w = 0.0f, s_a[NT][2];
            if constexpr (kBlock) {
                s_w = warp_ok ? __ldg(sseg + (size_t)(lrow0 >> 7) * a.kb + kb) : 0.0f;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t t0 = nt * 8 + t, t1 = t0 + 4;
                    s_a[nt][0] = t0 < a.m ? __ldg(a.sa + (size_t)t0 * a.kb + kb) : 0.0f;
                    s_a[nt][1] = t1 < a.m ? __ldg(a.sa + (size_t)t1 * a.kb + kb) : 0.0f;
                }
            }
            if (!*abort_flag && !mbar_wait(&full[slot], ph, a.wait_limit_ns)) fault(2);
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[nt][j] = 0.0f;
            const uint32_t wbox = smem_base + slot * L::kStage + warp * kWBox;
            const uint32_t abox = smem_base + slot * L::kStage + kWBytes;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t sw = ((uint32_t)((4 * c + t) ^ pg)) << 4;
                const uint4 A0 = lds128(wbox + pg * 128 + sw);
                const uint4 A1 = lds128(wbox + (8 + pg) * 128 + sw);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 B = lds128(abox + (nt * 8 + pg) * 128 + sw);
                    mma_e4m3_16832(acc[nt], A0.x, A1.x, A0.y, A1.y, B.x, B.y);
                    mma_e4m3_16832(acc[nt], A0.z, A1.z, A0.w, A1.w, B.z, B.w);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if constexpr (kBlock) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float s0 = s_a[nt][0] * s_w, s1 = s_a[nt][1] * s_w;
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
        }
        if constexpr (!kBlock) {  // per-row scales: sa[token] * sw[row]
            const bool ok0 = row0 + pg < a.n, ok1 = row0 + 8 + pg < a.n;
            const float w0 = ok0 ? __ldg(sseg + lrow0 + pg) : 0.0f;
            const float w1 = ok1 ? __ldg(sseg + lrow0 + 8 + pg) : 0.0f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t t0 = nt * 8 + t, t1 = t0 + 4;
                const float a0 = t0 < a.m ? __ldg(a.sa + t0) : 0.0f;
                const float a1 = t1 < a.m ? __ldg(a.sa + t1) : 0.0f;
                total[nt][0] *= a0 * w0;
                total[nt][1] *= a1 * w0;
                total[nt][2] *= a0 * w1;
                total[nt][3] *= a1 * w1;
            }
        }
    }

    // after a timeout, wait (bounded) for the copies still in flight
    __syncthreads();
    if (*abort_flag && warp == kConsumers && lane == 0) {
        const uint32_t first = issued > (uint32_t)kStages ? issued - kStages : 0;
        for (uint32_t it = first; it < issued; ++it)
            if (it != a.debug_skip_iter) mbar_wait(&full[it % kStages], (it / kStages) & 1, a.wait_limit_ns);
    }

    auto store = [&](uint32_t tok, uint32_t row, float v) {
        if (tok < a.m && row < a.n) {
            if (a.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)tok * a.ldc + row] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float *>(a.out)[(size_t)tok * a.ldc + row] = v;
        }
    };

    const int g = lane >> 2, t = lane & 3, pg = perm8(g);
    if (split == 1) {
        if (warp < kConsumers) {
            const uint32_t r0 = tile_row0 + 16 * warp + pg, r1 = r0 + 8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t t0 = nt * 8 + t, t1 = t0 + 4;
                store(t0, r0, total[nt][0]);
                store(t1, r0, total[nt][1]);
                store(t0, r1, total[nt][2]);
                store(t1, r1, total[nt][3]);
            }
        }
        return;
    }

    // split-K across the cluster: partials to shared memory, then CTA r sums
    // rows [r*128/split, (r+1)*128/split) over all ranks in rank order
    if (warp < kConsumers) {
        const int lr0 = 16 * warp + pg, lr1 = lr0 + 8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int t0 = nt * 8 + t, t1 = t0 + 4;
            red[t0 * kRowsPerCta + lr0] = total[nt][0];
            red[t1 * kRowsPerCta + lr0] = total[nt][1];
            red[t0 * kRowsPerCta + lr1] = total[nt][2];
            red[t1 * kRowsPerCta + lr1] = total[nt][3];
        }
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const uint32_t r_lo = (kRowsPerCta * sidx) / split, r_hi = (kRowsPerCta * (sidx + 1)) / split;
    const uint32_t span = r_hi - r_lo;
    for (uint32_t idx = threadIdx.x; idx < span * L::kActRows; idx += blockDim.x) {
        const uint32_t tok = idx / span, lrow = r_lo + idx % span;
        float sum = 0.0f;
        float v[8];
#pragma unroll
        for (int rk = 0; rk < 8; ++rk)
            v[rk] = rk < (int)split ? cluster.map_shared_rank(red, rk)[tok * kRowsPerCta + lrow] : 0.0f;
#pragma unroll
        for (int rk = 0; rk < 8; ++rk) sum += v[rk];  // rank order; absent ranks add +0
        store(tok, tile_row0 + lrow, sum);
    }
    cluster.sync();
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int NT, bool kBlock>
const uint32_t *cta_slots() {
    static std::mutex mu;
    static std::vector<std::vector<uint32_t>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    if (cache[dev].empty()) {
        const void *f = (const void *)w8a8_gemv_tma_kernel<NT, kBlock>;
        cudaFuncSetAttribute(w8a8_gemv_tma_kernel<NT, kBlock>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Layout<NT>::kAlloc);
        cache[dev].assign(8, 0);
        resident_cta_slots(f, kThreads, Layout<NT>::kAlloc, resident_ctas(f, kThreads, Layout<NT>::kAlloc, 0),
                           cache[dev].data());
    }
    return cache[dev].data();
}

}  // namespace

// Split of K over a cluster of CTAs.  Work is in 128-blocks; a CTA of split s
// takes up to ceil(kb/s) of them plus about two blocks' worth of pipeline
// fill and drain.  slots[s-1] CTAs of clusters of s can be resident at once.
// Choose s in 1..8 that minimises waves x per-CTA work, with a small charge
// for the cluster reduction.
uint32_t choose_split_k(uint32_t tiles, uint32_t kb, const uint32_t *slots, double reduce_cost) {
#ifdef QDL_TUNE_SPLIT
    if (QDL_TUNE_SPLIT > 0) return QDL_TUNE_SPLIT < kb ? QDL_TUNE_SPLIT : kb;
#endif
    uint32_t best = 1;
    double best_cost = 1e300;
    for (uint32_t s = 1; s <= 8 && s <= kb; ++s) {
        const uint32_t fit = slots[s - 1] >= s ? slots[s - 1] : s;
        const uint32_t units = tiles * s;
        const uint32_t waves = (units + fit - 1) / fit;
        const double cost =
            (double)waves * (((kb + s - 1) / s) + 2.0 + (s > 1 ? reduce_cost : 0.0)) * (1.0 + 0.03 * (s - 1));
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// CTAs that can be resident at once when launched in clusters of s = 1..8.
// With one CTA per SM the cluster occupancy query is used, since clusters must
// fit inside one GPC; with several per SM the SM count times CTAs per SM.
void resident_cta_slots(const void *func, int threads, size_t smem, int per_sm, uint32_t *out) {
    const uint32_t flat = (uint32_t)(device_sm_count() * (per_sm > 0 ? per_sm : 1));
    for (int s = 1; s <= 8; ++s) {
        uint32_t fit = flat / s * s;
        if (per_sm <= 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, s, 1);
            cfg.blockDim = dim3(threads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = s;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) == cudaSuccess && n > 0 && (uint32_t)(n * s) < fit)
                fit = (uint32_t)(n * s);
            cudaGetLastError();
        }
        out[s - 1] = fit;
    }
}

namespace {

template <int NT, bool kBlock>
cudaError_t launch_variant(const W8A8Args &a, const CUtensorMap (&maps)[4], cudaStream_t s) {
    const uint32_t tiles = (a.n + kRowsPerCta - 1) / kRowsPerCta;
    const uint32_t split = choose_split_k(tiles, a.kb, cta_slots<NT, kBlock>(), 0.0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, split, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Layout<NT>::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w8a8_gemv_tma_kernel<NT, kBlock>, maps[0], maps[1], maps[2], maps[3], a);
}

}  // namespace

// CTAs of a kernel that fit on one SM at once: shared memory (with the per-CTA
// reservation), threads, registers and tensor-memory columns (512 per SM).
int resident_ctas(const void *func, int threads, size_t smem, int tmem_cols) {
    int dev = 0, smem_sm = 0, reserved = 0, threads_sm = 0, regs_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
    cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    cudaFuncAttributes fa = {};
    cudaFuncGetAttributes(&fa, func);
    int n = smem_sm > 0 ? smem_sm / (int)(smem + reserved) : 1;
    if (threads_sm > 0) n = n < threads_sm / threads ? n : threads_sm / threads;
    const int regs_cta = ((fa.numRegs > 0 ? fa.numRegs : 32) + 7) / 8 * 8 * threads;
    if (regs_sm > 0) n = n < regs_sm / regs_cta ? n : regs_sm / regs_cta;
    if (tmem_cols > 0) n = n < 512 / tmem_cols ? n : 512 / tmem_cols;
    return n < 1 ? 1 : n;
}

cudaError_t make_tmap_u8(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t stride,
                         uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {stride};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// One launch for up to 16 token rows.  `segs` are the weight segments
// (pointer, rows); the tensor maps are built here.
cudaError_t launch_w8a8_gemv_tma(const W8A8Args &a, int format, const uint8_t *const seg_w[3],
                                 const uint32_t seg_n[3], cudaStream_t s) {
    CUtensorMap maps[4];
    for (int i = 0; i < 3; ++i) {
        cudaError_t e = make_tmap_u8(&maps[i], seg_w[i], a.k, seg_n[i], a.k, 128, 16);
        if (e != cudaSuccess) return e;
    }
    const uint32_t act_rows = a.m <= 8 ? 8 : 16;
    cudaError_t e = make_tmap_u8(&maps[3], a.q, a.k, a.m, a.k, 128, act_rows);
    if (e != cudaSuccess) return e;
    const bool blk = format == QDL_SCALE_BLOCK128;
    if (a.m <= 8) return blk ? launch_variant<1, true>(a, maps, s) : launch_variant<1, false>(a, maps, s);
    return blk ? launch_variant<2, true>(a, maps, s) : launch_variant<2, false>(a, maps, s);
}

cudaError_t plan_w8a8_gemv_tma(const W8A8Args &a, int format, PlanInfo *p) {
    const bool blk = format == QDL_SCALE_BLOCK128;
    const uint32_t *slots = a.m <= 8 ? (blk ? cta_slots<1, true>() : cta_slots<1, false>())
                                     : (blk ? cta_slots<2, true>() : cta_slots<2, false>());
    p->kernel = 1;
    p->mma_n = a.m <= 8 ? 8 : 16;
    p->tiles = (a.n + kRowsPerCta - 1) / kRowsPerCta;
    p->split = choose_split_k(p->tiles, a.kb, slots, 0.0);
    p->stages = kStages;
    p->threads = kThreads;
    p->smem = a.m <= 8 ? Layout<1>::kAlloc : Layout<2>::kAlloc;
    p->clusters = (int)(slots[p->split - 1] / p->split);
    return cudaGetLastError();
}

cudaError_t read_and_clear_gemv_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_gemv_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_gemv_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
