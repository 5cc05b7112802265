// Host-side helpers shared by the kernels' launchers: TMA tensor-map
// encoding (through the driver's cuTensorMapEncodeTiled, looked up once),
// per-SM residency of a kernel, and the split-K choice of the tcgen05 GEMV.
#include <mutex>

#include "tma_pipe.cuh"

namespace qdl {

namespace {

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

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t outer,
                      uint64_t stride, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {inner, outer};
    cuuint64_t gstride[1] = {stride};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, type, 2, const_cast<void *>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t make_tmap_u8(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t stride,
                         uint32_t box_cols, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, cols, rows, stride, box_cols, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t make_tmap_4b(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    return encode_2d(map, type, base, inner, outer, inner * 4, box_inner, box_outer, swizzle);
}

cudaError_t make_tmap_plain(CUtensorMap *map, bool f32, const void *base, uint64_t inner, uint64_t outer,
                            uint32_t box_inner, uint32_t box_outer) {
    return make_tmap_4b(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT32, base, inner, outer,
                        box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t make_tmap_words(CUtensorMap *map, const void *base, uint64_t words, uint64_t rows, uint32_t box_rows) {
    return make_tmap_4b(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, base, words, rows, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t make_tmap_f32(CUtensorMap *map, const float *x, uint64_t k, uint64_t rows, uint32_t box_rows) {
    return make_tmap_4b(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, k, rows, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

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

}  // namespace qdl
