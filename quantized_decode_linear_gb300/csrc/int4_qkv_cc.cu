// AWQ INT4 fused Q/K/V projection for a few token rows on the CUDA cores
// (fused_int4_qkv.rs: fused_int4_qkv_q, fused_int4_qkv_k, fused_int4_qkv_v,
// unpack_awq_qkv, QKV_AWQ_SHIFTS).  One launch covers all three projections,
// up to 4 token rows.
//
// With one to a few tokens every weight is used once or a few times, so the
// work is a stream of 4-bit codes: this kernel keeps them in a deep TMA ring
// and spends about two ALU operations per code on turning it into an exact
// f32, plus one FMA per token.
//
// Arithmetic (per group g, column c, token t):
//   y[t, c] = sum_g s[g,c] ( sum_{k in g} x[t,k] nib[k,c] - z[g,c] sum_{k in g} x[t,k] )
// which is sum_k x (nib - z) s regrouped; x stays f32, nib is exact, the inner
// sums accumulate in f32.  A nibble at bit 4e of a word (e <= 4) becomes the
// float nib * 16^e exactly: OR its masked bits into the pattern of 2^23 and
// subtract 2^23.  The 16^-e factor is applied to s at the group's end, where
// it is exact (a power of two).  The AWQ word holds columns
// {0, 2, 4, 6, 1, 3, 5, 7} at nibbles 0..7 (shifts {0,16,4,20,8,24,12,28} of
// columns 0..7); nibbles 5..7 are read from the word shifted right by 12.
//
// Roles (one CTA = 256 output columns of one projection x a range of groups;
// one stage = 64 K rows):
//   warp 0, one lane : TMA producer: the stage's [64 rows x 32 words] of
//                      packed codes (128-byte rows, 128-byte swizzle) and the
//                      two [tokens x 32] boxes of x, into a ring of stages.
//   warps 1..C       : consumers (C = 16 for up to 2 tokens, else 8).  Warp w
//                      takes 64/C consecutive rows of each stage; lane l owns
//                      word column l (8 output columns) and keeps, per token,
//                      a running sum for the group and the folded total.
// The consumer warps' totals are added in shared memory in warp order, and the
// split-K CTAs of one cluster add theirs through distributed shared memory in
// rank order.  Every wait is bounded (fault word, drain, return).
#include <cooperative_groups.h>

#include <mutex>
#include <vector>

#include "tma_pipe.cuh"

namespace cg = cooperative_groups;

namespace qdl {

static __device__ uint32_t g_int4cc_fault;

namespace {

constexpr int kColsC = 256;                              // output columns per CTA (32 words)
constexpr int kRowsC = 64;                               // K rows per stage
constexpr uint32_t kWordBytes = kRowsC * 128;            // 8 KB of packed codes
constexpr uint32_t kXSlot = 1024;                        // one x box: up to 4 tokens x 32 f32 (1 KB apart)
constexpr uint32_t kStageC = kWordBytes + 2 * kXSlot;    // multiple of 1024 (swizzle atoms)
constexpr int kRingC = 16;
constexpr uint32_t kBarOffC = kRingC * kStageC;
constexpr uint32_t kAllocC = kBarOffC + 512 + 1024;
static_assert((2 * kRingC + 2) * 8 <= 512, "barrier area");
static_assert(16 * 4 * kColsC * 4 + 4 * kColsC * 4 <= kBarOffC, "reduction areas fit in the ring");

// consumer warps: 16 (4 rows of a stage each) for up to 2 tokens, where
// more warps hide latency; 8 (8 rows each) for more tokens, whose register
// needs allow fewer warps
template <int MT>
struct Cc {
    static constexpr int kConsumers = MT <= 2 ? 16 : 8;
    static constexpr int kRowsW = kRowsC / kConsumers;  // rows of a stage per consumer warp
    static constexpr int kThreads = (1 + kConsumers) * 32;
};

// column (within the word) held by physical nibble p, and the exponent e of
// the value nib * 16^e that nibble p is read as
__device__ __forceinline__ constexpr int nib_col(int p) { return p < 4 ? 2 * p : 2 * (p - 4) + 1; }
__device__ __forceinline__ constexpr int nib_exp(int p) { return p <= 4 ? p : p - 3; }

// exact f32 value nib * 16^e of the nibble at bits [4e, 4e+4) of v (e <= 4)
__device__ __forceinline__ float nib_scaled(uint32_t v, int e) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0xFu << (4 * e)), "r"(0x4B000000u));  // (v & m) | c
    return __uint_as_float(r) - 8388608.0f;
}

template <int MT>
__global__ void __launch_bounds__(Cc<MT>::kThreads, 1)
    int4_qkv_cc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_x,
                       const Int4Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kBarOffC);  // [kRingC] codes and x landed
    uint64_t *empty = full + kRingC;                                 // [kRingC] every consumer done
    volatile uint32_t *abort_flag = reinterpret_cast<uint32_t *>(empty + kRingC);
    constexpr int kConsumers = Cc<MT>::kConsumers, kRowsW = Cc<MT>::kRowsW;
    float *red = reinterpret_cast<float *>(smem);                          // [kConsumers][MT][256] at the end
    float *part = reinterpret_cast<float *>(smem) + kConsumers * MT * kColsC;  // [MT][256]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // projection and column tile of this CTA
    uint32_t tile = blockIdx.x;
    const CUtensorMap *tmap;
    const float *sc, *zr;
    float *out;
    uint32_t n;
    if (tile < a.tiles_q) {
        tmap = &tm_q; sc = a.sc0; zr = a.zr0; out = a.out0; n = a.nq;
    } else if (tile < a.tiles_q + a.tiles_kv) {
        tile -= a.tiles_q;
        tmap = &tm_k; sc = a.sc1; zr = a.zr1; out = a.out1; n = a.nkv;
    } else {
        tile -= a.tiles_q + a.tiles_kv;
        tmap = &tm_v; sc = a.sc2; zr = a.zr2; out = a.out2; n = a.nkv;
    }
    const uint32_t col0 = tile * kColsC;
    const uint32_t split = gridDim.y, sidx = blockIdx.y;
    const uint32_t row_lo = ((a.groups * sidx) / split) * a.group;
    const uint32_t row_hi = ((a.groups * (sidx + 1)) / split) * a.group;
    const uint32_t nstage = (row_hi - row_lo + kRowsC - 1) / kRowsC;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingC; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    auto fault = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(&g_int4cc_fault, code);
    };
    auto wait = [&](uint64_t *bar, uint32_t parity, uint32_t code) {
        if (!*abort_flag && !mbar_wait(bar, parity, kWaitLimitNs)) fault(code);
    };

    uint32_t issued = 0;
    float y[8][MT];  // folded totals, by physical nibble
#pragma unroll
    for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int t = 0; t < MT; ++t) y[p][t] = 0.0f;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(tmap);
            prefetch_tmap(&tm_x);
            const uint64_t pol = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            constexpr uint32_t kTx = kWordBytes + 2 * MT * 128;
            // codes of the first stages before waiting for the previous kernel
            const uint32_t head = nstage < (uint32_t)kRingC ? nstage : (uint32_t)kRingC;
            for (uint32_t st = 0; st < head; ++st) {
                mbar_arrive_expect_tx(&full[st], kTx);
                issued = st + 1;
                tma_load_2d(smem + st * kStageC, tmap, (int32_t)(col0 / 8), (int32_t)(row_lo + st * kRowsC), &full[st],
                            pol);
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");  // x is written by the previous kernel
            for (uint32_t st = 0; st < head; ++st) {
                const int32_t k0 = (int32_t)(row_lo + st * kRowsC);
                tma_load_2d(smem + st * kStageC + kWordBytes, &tm_x, k0, 0, &full[st], pol_x);
                tma_load_2d(smem + st * kStageC + kWordBytes + kXSlot, &tm_x, k0 + 32, 0, &full[st], pol_x);
            }
            for (uint32_t st = head; st < nstage; ++st) {
                const uint32_t slot = st % kRingC, ph = (st / kRingC) & 1;
                wait(&empty[slot], ph ^ 1, 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], kTx);
                issued = st + 1;
                uint8_t *stg = smem + slot * kStageC;
                const int32_t k0 = (int32_t)(row_lo + st * kRowsC);
                tma_load_2d(stg, tmap, (int32_t)(col0 / 8), k0, &full[slot], pol);
                tma_load_2d(stg + kWordBytes, &tm_x, k0, 0, &full[slot], pol_x);
                tma_load_2d(stg + kWordBytes + kXSlot, &tm_x, k0 + 32, 0, &full[slot], pol_x);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;
        const uint32_t wcol = col0 / 8 + lane;  // this lane's word column
        const bool col_ok = wcol < n / 8;
        float acc[8][MT], sx[MT];
#pragma unroll
        for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[p][t] = 0.0f;
#pragma unroll
        for (int t = 0; t < MT; ++t) sx[t] = 0.0f;
        float4 s_lo = make_float4(0, 0, 0, 0), s_hi = s_lo, z_lo = s_lo, z_hi = s_lo;
        uint32_t gcur = 0xFFFFFFFFu;

        // s (acc / 16^e - z sum x) of the group just finished into y
        auto fold = [&]() {
            const float s8[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
            const float z8[8] = {z_lo.x, z_lo.y, z_lo.z, z_lo.w, z_hi.x, z_hi.y, z_hi.z, z_hi.w};
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float s = s8[nib_col(p)];
                const float se = s * (1.0f / (float)(1u << (4 * nib_exp(p))));  // exact: a power of two
                const float zs = z8[nib_col(p)] * s;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    y[p][t] = fmaf(se, acc[p][t], y[p][t]);
                    y[p][t] = fmaf(-zs, sx[t], y[p][t]);
                    acc[p][t] = 0.0f;
                }
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) sx[t] = 0.0f;
        };

        for (uint32_t st = 0; st < nstage; ++st) {
            const uint32_t slot = st % kRingC, ph = (st / kRingC) & 1;
            wait(&full[slot], ph, 2);
            if (*abort_flag) break;
            const uint32_t sr0 = kRowsW * cw;              // first row of this warp's slice in the stage
            const uint32_t r0 = row_lo + st * kRowsC + sr0;  // and its K row
            if (r0 < row_hi) {
                const uint32_t g = r0 / a.group;  // the slice lies in one group (group % 16 == 0)
                if (g != gcur) {
                    if (gcur != 0xFFFFFFFFu) fold();
                    gcur = g;
                    if (col_ok) {
                        const float4 *sp = reinterpret_cast<const float4 *>(sc + (size_t)g * n + 8 * wcol);
                        const float4 *zp = reinterpret_cast<const float4 *>(zr + (size_t)g * n + 8 * wcol);
                        s_lo = __ldg(sp); s_hi = __ldg(sp + 1);
                        z_lo = __ldg(zp); z_hi = __ldg(zp + 1);
                    }
                }
                const uint8_t *stg = smem + slot * kStageC;
                // x of this slice: box sr0 / 32, 16-byte chunks (sr0 % 32) / 4 .. of each token row
                const uint8_t *xb = stg + kWordBytes + (sr0 >> 5) * kXSlot;
#pragma unroll
                for (int q = 0; q < kRowsW / 4; ++q) {  // rows 4q .. 4q+3 of the slice: one chunk of x
                    const uint32_t ch = ((sr0 & 31) >> 2) + q;
                    float xr[MT][4];
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const float4 v = *reinterpret_cast<const float4 *>(xb + t * 128 + ((ch ^ (t & 7)) << 4));
                        xr[t][0] = v.x; xr[t][1] = v.y; xr[t][2] = v.z; xr[t][3] = v.w;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t r = sr0 + 4 * q + i;  // row within the stage
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(
                            stg + r * 128 + ((((uint32_t)lane >> 2) ^ (r & 7)) << 4) + ((lane & 3) << 2));
                        const uint32_t h = w >> 12;
                        float f[8];
#pragma unroll
                        for (int p = 0; p < 8; ++p) f[p] = nib_scaled(p <= 4 ? w : h, nib_exp(p));
#pragma unroll
                        for (int t = 0; t < MT; ++t) {
#pragma unroll
                            for (int p = 0; p < 8; ++p) acc[p][t] = fmaf(xr[t][i], f[p], acc[p][t]);
                            sx[t] += xr[t][i];
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        if (gcur != 0xFFFFFFFFu) fold();
    }

    // ---------------------------------------------------------------- drain after a timeout
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t first = issued > (uint32_t)kRingC ? issued - kRingC : 0;
            for (uint32_t st = first; st < issued; ++st) mbar_wait(&full[st % kRingC], (st / kRingC) & 1, kWaitLimitNs);
        }
        __syncthreads();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs may be read or written by earlier kernels

    // ---------------------------------------------------------------- reduction
    // warps in order, then (split > 1) cluster ranks in order
    if (warp >= 1) {
#pragma unroll
        for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int t = 0; t < MT; ++t) red[((warp - 1) * MT + t) * kColsC + 8 * lane + nib_col(p)] = y[p][t];
    }
    __syncthreads();
    const uint32_t m_used = a.m < (uint32_t)MT ? a.m : (uint32_t)MT;
    for (uint32_t idx = threadIdx.x; idx < m_used * kColsC; idx += blockDim.x) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) s += red[w * MT * kColsC + idx];
        const uint32_t t = idx / kColsC, c = idx % kColsC;
        if (split == 1) {
            if (col0 + c < n) out[(size_t)t * n + col0 + c] = s;
        } else {
            part[idx] = s;
        }
    }
    if (split > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const uint32_t c_lo = (kColsC * sidx) / split, c_hi = (kColsC * (sidx + 1)) / split;
        const uint32_t span = c_hi - c_lo;
        const float *peer[8];
#pragma unroll
        for (int rk = 0; rk < 8; ++rk) peer[rk] = cluster.map_shared_rank(part, rk < (int)split ? rk : 0);
        for (uint32_t idx = threadIdx.x; idx < span * m_used; idx += blockDim.x) {
            const uint32_t t = idx / span, c = c_lo + idx % span;
            float v[8];
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) v[rk] = rk < (int)split ? peer[rk][t * kColsC + c] : 0.0f;
            float s = 0.0f;
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) s += v[rk];  // rank order; absent ranks add +0
            if (col0 + c < n) out[(size_t)t * n + col0 + c] = s;
        }
        cluster.sync();  // no rank leaves while others still read its partials
    }
}

template <int MT>
const uint32_t *cluster_fit_cc() {
    static std::mutex mu;
    static std::vector<std::vector<uint32_t>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    if (cache[dev].empty()) {
        const void *f = (const void *)int4_qkv_cc_kernel<MT>;
        cudaFuncSetAttribute(int4_qkv_cc_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAllocC);
        const int per_sm = resident_ctas(f, Cc<MT>::kThreads, kAllocC, 0);
        cache[dev].assign(8, 0);
        resident_cta_slots(f, Cc<MT>::kThreads, kAllocC, per_sm, cache[dev].data());
    }
    return cache[dev].data();
}

template <int MT>
cudaError_t launch_cc(const Int4Args &a, const CUtensorMap (&maps)[4], cudaStream_t s) {
    const uint32_t tiles = a.tiles_q + 2 * a.tiles_kv;
    const uint32_t split = choose_split_k(tiles, a.groups, cluster_fit_cc<MT>(), 0.0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, split, 1);
    cfg.blockDim = dim3(Cc<MT>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = kAllocC;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = split;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, int4_qkv_cc_kernel<MT>, maps[0], maps[1], maps[2], maps[3], a);
}

}  // namespace

bool int4_cc_supported(uint32_t nq, uint32_t nkv) { return nq % 32 == 0 && nkv % 32 == 0; }

cudaError_t launch_int4_qkv_cc(const Int4Args &a, cudaStream_t s) {
    if (a.m < 1 || a.m > 4) return cudaErrorInvalidValue;
    CUtensorMap maps[4];
    const uint32_t ns[3] = {a.nq, a.nkv, a.nkv};
    const uint32_t *qw[3] = {a.qw0, a.qw1, a.qw2};
    for (int p = 0; p < 3; ++p) {
        cudaError_t e = make_tmap_words(&maps[p], qw[p], ns[p] / 8, a.k, kRowsC);
        if (e != cudaSuccess) return e;
    }
    const uint32_t mt = a.m <= 1 ? 1 : a.m <= 2 ? 2 : 4;
    cudaError_t e = make_tmap_f32(&maps[3], a.x, a.k, a.m, mt);
    if (e != cudaSuccess) return e;
    Int4Args b = a;  // this kernel's tiles are 256 columns wide
    b.tiles_q = (a.nq + kColsC - 1) / kColsC;
    b.tiles_kv = (a.nkv + kColsC - 1) / kColsC;
    switch (mt) {
        case 1: return launch_cc<1>(b, maps, s);
        case 2: return launch_cc<2>(b, maps, s);
        default: return launch_cc<4>(b, maps, s);
    }
}

cudaError_t read_and_clear_int4cc_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_int4cc_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_int4cc_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
