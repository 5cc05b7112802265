// W8A8 decode GEMV / skinny GEMM on the 5th-generation tensor cores
// (w8a8_decode.rs fn w8a8_gemv and fn w8a8_proj; segment routing from
// W8a8Weight::boundaries; scale layouts from enum W8a8Scale).  One pass over
// the weights for any token count (token blocks of 256 beyond 256 rows).
//
//   y[m, j] = sum_kb Sa(m, kb) Sw(j, kb) sum_{k in kb} dec(q[m,k]) dec(W[j,k])
//
// Roles (one CTA = 128 output rows x a range of 128-wide K blocks):
//   warp 0, one lane : TMA producer.  Per K block, the 128 x 128-byte weight
//                      tile (one box, or eight 16-row boxes when the tile
//                      spans two segments) and the NTOK-row activation box
//                      land in a shared-memory stage (128-byte
//                      swizzle = the canonical K-major SW128 operand layout).
//   warp 1           : allocates the tensor memory; one lane issues
//                      tcgen05.mma kind::f8f6f4 (M = 128 weight rows,
//                      N = NTOK tokens, K = 32 per instruction, four per
//                      block) and commits each stage back to its `empty`
//                      mbarrier.
//   warp 2 (Block128): copies the raw scales of the next K blocks in with
//                      cp.async and stages sa[m, kb] * sw[kb] for each block
//                      in shared memory for the epilogue (one buffer per
//                      accumulator).
//   other warps      : epilogue, reading the f32 accumulators with tcgen05.ld.
//
// Scales.  PerRow: the accumulator sums the CTA's whole K range; the epilogue
// multiplies by sa[m] sw[j].  Block128: each 128-block accumulates into one of
// 2-4 TMEM buffers in turn; the epilogue folds a finished buffer into
// register totals with sa[m, kb] sw[j/128, kb] (packed f32x2 FMAs) while the
// tensor core fills the next ones.  At the end the totals go through the
// freed stage ring as [token][row] and leave in 16-byte pieces.
//
// Launch overlap.  Kernels are launched with programmatic stream
// serialisation: the weight stream (independent of earlier kernels) starts at
// once; every read of activations or scales and every output write comes
// after griddepcontrol.wait.
//
// Split-K CTAs of one cluster reduce their partials through distributed shared
// memory in rank order (deterministic), or, when the caller has zeroed an f32
// output (the projection entry points), add them into it with f32 reductions
// (no cluster barrier; the order of the additions varies from run to run).
// Every wait is bounded; after a timeout the CTA records a fault word, waits
// (bounded) for its copies and MMAs in flight, frees its tensor memory and
// returns.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <mutex>
#include <vector>

#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

#ifndef QDL_TC_MIN_STAGES
#define QDL_TC_MIN_STAGES 3
#endif
#ifndef QDL_TC_EARLY_TRIGGER_BYTES
// A 16-token GEMV over at least this many weight bytes releases its dependent
// kernels as soon as it starts (before its own dependency wait it only
// streams read-only weights), so that the next call's kernels launch while
// this one streams.  Measured: 38.1 -> 36.6 us on the K=8192, N=28672 gate/up
// projection at M=1.  On the 25 MB QKV projection at M=8 it pays only with
// the 3-stage ring below (8.01 -> 7.58 us per call): with 4 stages, 3 CTAs
// per SM, the next call's CTAs found almost no free slot and the call slowed
// (7.7 -> 8.0 us).
#define QDL_TC_EARLY_TRIGGER_BYTES (16ull << 20)
#endif
#ifndef QDL_TC_EARLY_MAX_NTOK
#define QDL_TC_EARLY_MAX_NTOK 16  // token buckets that release their dependents at the start
#endif
#ifndef QDL_TC_STAGE_BYTES_16
// the 16-token variants: 3 stages of 18 KB.  With the scale staging a CTA
// needs 57.4 KB (58.4 KB with the driver's reservation), so 3 share an SM; a
// 256-byte smaller barrier area fits 4, which measured faster for the 25 MB
// QKV projection at M = 8 (GEMV 5.82 -> 5.01 us) but slower for the 235 MB
// gate/up projection at M = 1-16 (0.5-1 us per call), and requesting padded
// shared memory for wide launches to keep those at 3 slowed its 16-row calls
#define QDL_TC_STAGE_BYTES_16 (54 * 1024)
#endif
#ifndef QDL_TC_STAGE_BYTES
#define QDL_TC_STAGE_BYTES (72 * 1024)
#endif
// ... and for the wide variants (NTOK >= QDL_TC_BIG_NTOK) that run one CTA per SM
#ifndef QDL_TC_STAGE_BYTES_BIG
#define QDL_TC_STAGE_BYTES_BIG (72 * 1024)
#endif
// token buckets in which the accumulating Block128 GEMV runs stream-K (a
// 256-token stream-K variant spilled at its 96-register budget and measured
// 2.6x slower than the split-K launch)
// ... and for the Block128 64- and 128-token variants (the stream-K GEMV of
// the f32 projection among them).  128 tokens: one CTA per SM with 4 stages
// of 32 KB took the K=8192, N=28672 gate/up projection at M=128 from 77.0 to
// 72.2 us (6 stages 75.4).  64 tokens: 3 stages of 24 KB with the registers
// capped at 128, so that 2 CTAs share an SM, took M=64 from 52.8 to 47.0 us
// per call against one CTA of 7 stages at 210 registers (2 CTAs of 4
// stages: 54.7).  Deeper rings measured no better for the 32-token variant
// (48.0 vs 48.4 us at M=32) and slower for the per-row and 256-token variants.
#ifndef QDL_TC_STAGE_BYTES_B128
#define QDL_TC_STAGE_BYTES_B128 (144 * 1024)
#endif
#ifndef QDL_TC_STAGE_BYTES_B64
#define QDL_TC_STAGE_BYTES_B64 (72 * 1024)
#endif
#ifndef QDL_TC_ADD_NOCLUSTER
#define QDL_TC_ADD_NOCLUSTER 1
#endif
#ifndef QDL_STREAMK_MIN_NTOK
#define QDL_STREAMK_MIN_NTOK 32
#endif
#ifndef QDL_STREAMK_MAX_NTOK
#define QDL_STREAMK_MAX_NTOK 128
#endif
#ifndef QDL_TC_BIG_NTOK
#define QDL_TC_BIG_NTOK 128
#endif
// Block128 epilogue: accumulator columns read from tensor memory per wait
// (loads in flight), and register caps that let several CTAs share an SM
#ifndef QDL_TC_INFLIGHT_SMALL
#define QDL_TC_INFLIGHT_SMALL 32  // NTOK <= 64
#endif
#ifndef QDL_TC_INFLIGHT_128
#define QDL_TC_INFLIGHT_128 64
#endif
#ifndef QDL_TC_INFLIGHT_256
#define QDL_TC_INFLIGHT_256 16
#endif
#ifndef QDL_TC_REGS_32
// 80: 3 CTAs of 7 warps fit an SM (6 warps on some sub-partition); at 96 only
// 2 fit.  Despite a small spill, 3 per SM in one even wave took the gate/up
// projection at M = 32 from 43.9 to 40.3 us per call (2 per SM in three waves)
#define QDL_TC_REGS_32 80
#endif
#ifndef QDL_TC_EPI_256
#define QDL_TC_EPI_256 16  // epilogue warps of the 256-token Block128 variant
#endif
#ifndef QDL_TC_REGS_64
#define QDL_TC_REGS_64 128  // 2 CTAs of 7 warps per SM (a small spill in the stream-K variant)
#endif
#ifndef QDL_TC_REGS_256
#define QDL_TC_REGS_256 104  // one CTA of 19 warps: all the registers it can have
#endif
#ifndef QDL_TC_ACC_128
// accumulator buffers of the 128-token Block128 variants (4 and 2 measured
// the same on the gate/up projection at M = 128: 62.2 and 62.3 us per call)
#define QDL_TC_ACC_128 4
#endif
#ifndef QDL_TC_SCALE_AHEAD
// K blocks whose scales the Block128 scale warp has in flight: its global
// reads wait out the memory latency of a loaded GPU (measured on the 256-row
// gate/up projection: the scale reads one block ahead cost ~10 us of 83)
#define QDL_TC_SCALE_AHEAD 4
#endif
#ifndef QDL_TC_FFMA2
// Block128 folds as packed f32x2 FMAs (0: scalar FMAs, same rounding): M = 128
// 85.9 -> 75.2 us and M = 256 103.5 -> 93.9 us per call with the 32x32b and
// 16x256b fragments respectively
#define QDL_TC_FFMA2 1
#endif
// token buckets from which the Block128 fold reads tensor memory in the
// 16x256b shape (see Tc::kFrag)
#ifndef QDL_TC_FRAG_MIN_NTOK
#define QDL_TC_FRAG_MIN_NTOK 128
#endif
#ifndef QDL_TC_BIGBOX
#define QDL_TC_BIGBOX 1
#endif

namespace qdl {

static __device__ uint32_t g_tc_fault;

namespace {

constexpr int kTileRows = 128;
constexpr uint32_t kWBytes = kTileRows * 128;  // weight tile per stage
constexpr uint32_t kWBox = 16 * 128;
// totals staged in the freed stage ring at the end: [token][kRedStride] floats
// (the 4-float pad puts the rows that one warp store covers in distinct banks)
constexpr uint32_t kRedStride = kTileRows + 4;

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
    static constexpr uint32_t kBudget = kBlock && NTOK == 128 ? QDL_TC_STAGE_BYTES_B128
                                        : kBlock && NTOK == 64  ? QDL_TC_STAGE_BYTES_B64
                                        : NTOK >= QDL_TC_BIG_NTOK ? QDL_TC_STAGE_BYTES_BIG
                                        : NTOK == 16              ? QDL_TC_STAGE_BYTES_16
                                                                  : QDL_TC_STAGE_BYTES;
    static constexpr int kMinStages = NTOK <= 64 ? QDL_TC_MIN_STAGES : 3;
    static constexpr int kStages = (int)(kBudget / kStage) < kMinStages ? kMinStages : (int)(kBudget / kStage);
    // Block128 accumulator buffers: the MMA may run kAcc-1 blocks ahead of
    // the epilogue that folds each block's scales
    static constexpr int kAcc = kBlock ? (NTOK <= 64 ? 4 : NTOK == 128 ? QDL_TC_ACC_128 : 2) : 1;
    static constexpr uint32_t kBarOff = kStages * kStage;
    static constexpr uint32_t kScaleOff = kBarOff + 512;  // Block128: [kAcc][kSBuf] block scales
    // Block128 epilogue fragments: 16x256b (a thread holds 4 rows x 2 token
    // columns per 8 columns) for NTOK >= QDL_TC_FRAG_MIN_NTOK, else 32x32b (one
    // row x every column).  The 16-lane shape reads tensor memory at about half
    // the rate (measured ~250 against >= 400 B/clk per SM) but needs a quarter
    // of the scale broadcasts, which pays only for wide token blocks.
    static constexpr bool kFrag = kBlock && NTOK >= QDL_TC_FRAG_MIN_NTOK;
    // Scales of one accumulator buffer in the order the fragments use them:
    // 32x32b, token t at [t]; 16x256b, token t at [(t % 8) / 2][2 (t / 8) + t % 2],
    // four rows of kSRow floats (padded by 16 bytes so that the four rows the
    // lanes of a quarter-warp read fall in different banks)
    static constexpr uint32_t kSRow = kFrag ? NTOK / 4 + 4 : NTOK;
    static constexpr uint32_t kSBuf = kFrag ? 4 * kSRow : NTOK;
    // Block128: raw activation scales of kSAhead K blocks ahead, copied in by
    // the scale warp ([kSAhead][kSStage]: NTOK tokens, then the block's weight scale)
    static constexpr int kSAhead = QDL_TC_SCALE_AHEAD;
    static constexpr uint32_t kSStage = NTOK + 4;
    static constexpr uint32_t kStageOff = kScaleOff + (kBlock ? kAcc * kSBuf * 4 : 0);
    static constexpr uint32_t kBytes = kStageOff + (kBlock ? kSAhead * kSStage * 4 : 0);
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static constexpr int kEpiBase = kBlock ? 3 : 2;                          // first epilogue warp
    static constexpr int kEpi = kBlock ? (NTOK <= 64 ? 4 : NTOK == 256 ? QDL_TC_EPI_256 : NTOK / 16) : 4;  // epilogue warps
    static constexpr int kCpt = kBlock ? NTOK * 4 / kEpi : 16;               // columns per epilogue thread
    static constexpr int kThreads = (kEpiBase + kEpi) * 32;
    // columns per tensor-memory wait in the Block128 epilogue
    static constexpr int kInFlight =
        kCpt < (NTOK <= 64 ? QDL_TC_INFLIGHT_SMALL : NTOK == 128 ? QDL_TC_INFLIGHT_128 : QDL_TC_INFLIGHT_256)
            ? kCpt
            : (NTOK <= 64 ? QDL_TC_INFLIGHT_SMALL : NTOK == 128 ? QDL_TC_INFLIGHT_128 : QDL_TC_INFLIGHT_256);
    // register cap per thread, so that several CTAs fit an SM (255: none):
    // 32 tokens 3 per SM, 64 tokens 2 per SM (warps per SM sub-partition x 32
    // x registers must stay within its 16K registers)
    static constexpr int kMaxRegs = !kBlock ? 255 : NTOK == 32 ? QDL_TC_REGS_32 : NTOK == 64 ? QDL_TC_REGS_64 : NTOK == 256 ? QDL_TC_REGS_256 : 255;
    static constexpr uint32_t kTmemCols = pow2_at_least(kAcc * NTOK);
    static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(NTOK * kRedStride * 4 <= kBarOff, "the staged totals must fit in the stage ring");
    static_assert(kTmemCols <= 512, "tensor memory");
    static_assert((2 * kStages + 3 * kAcc + 1) * 8 + 8 <= 512, "barrier area");
    static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
    static_assert(kInFlight % 16 == 0 && kCpt % kInFlight == 0, "epilogue load groups");
};

// ---------------------------------------------------------------- kernel helpers

// Block128 epilogue layout.  Epilogue warp e reads tensor-memory lanes
// 32 (warp % 4) .. +31 (weight rows) and token columns kCpt (e / 4) .. +kCpt-1.
// A thread's total j is the accumulator of
//   32x32b : token kCpt (e / 4) + j, row 32 (warp % 4) + lane
//   16x256b: token kCpt (e / 4) + 8 (j / 8) + 2 (lane % 4) + j % 2,
//            row   32 (warp % 4) + 16 ((j / 4) % 2) + 8 ((j / 2) % 2) + lane / 4
template <bool kFrag>
__device__ __forceinline__ uint32_t frag_tok(int j, uint32_t lane) {
    return kFrag ? 8u * (uint32_t)(j >> 3) + 2u * (lane & 3u) + (uint32_t)(j & 1) : (uint32_t)j;
}
template <bool kFrag>
__device__ __forceinline__ uint32_t frag_row(int j, uint32_t lane) {
    return kFrag ? 16u * (uint32_t)((j >> 2) & 1) + 8u * (uint32_t)((j >> 1) & 1) + (lane >> 2) : lane;
}
// position of token t's scale in one accumulator buffer's scale block
template <int NTOK>
__device__ __forceinline__ uint32_t scale_slot(uint32_t t) {
    using C = Tc<NTOK, true>;
    return C::kFrag ? ((t & 7u) >> 1) * C::kSRow + 2u * (t >> 3) + (t & 1u) : t;
}
// this thread's first scale in a buffer (epilogue column group cgrp)
template <int NTOK>
__device__ __forceinline__ uint32_t scale_row(uint32_t cgrp, uint32_t lane) {
    using C = Tc<NTOK, true>;
    return C::kFrag ? (lane & 3u) * C::kSRow + cgrp * C::kCpt / 4 : cgrp * C::kCpt;
}

// total[j, j+1] += (v0, v1) * (s0, s1) as one packed f32x2 FMA (each half
// rounded as the scalar fmaf would be)
__device__ __forceinline__ void fma_pair(float &t0, float &t1, float v0, float v1, float s0, float s1) {
#if QDL_TC_FFMA2
    const float2 r = __ffma2_rn(make_float2(v0, v1), make_float2(s0, s1), make_float2(t0, t1));
    t0 = r.x;
    t1 = r.y;
#else
    t0 = fmaf(v0, s0, t0);
    t1 = fmaf(v1, s1, t1);
#endif
}

// Fold the finished accumulator buffer at tensor-memory column `col_b` into
// the totals: total[j] += D[row(j), tok(j)] * s[tok(j)], with `sq` this
// thread's first scale (scale_row).
template <int NTOK>
__device__ __forceinline__ void fold_block(uint32_t taddr, uint32_t col_b, const float *sq,
                                           float (&total)[Tc<NTOK, true>::kCpt]) {
    using C = Tc<NTOK, true>;
    constexpr int kCpt = C::kCpt, kF = C::kInFlight;
#pragma unroll
    for (int g = 0; g < kCpt / kF; ++g) {
        if constexpr (C::kFrag) {
            float va[kF / 2], vb[kF / 2];  // lanes +0..15 and +16..31 of the warp's 32
            tc_ld_16x256b<kF / 8>(taddr + col_b + kF * g, va);
            tc_ld_16x256b<kF / 8>(taddr + (16u << 16) + col_b + kF * g, vb);
            tc_wait_ld();
            const float4 *sp = reinterpret_cast<const float4 *>(sq + kF / 4 * g);
#pragma unroll
            for (int q4 = 0; q4 < kF / 16; ++q4) {
                const float4 s4 = sp[q4];  // the scales of two 8-column chunks
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = 2 * q4 + h;  // chunk within the group
                    const float se = h ? s4.z : s4.x, so = h ? s4.w : s4.y;
                    float *t = total + kF * g + 8 * j;
                    fma_pair(t[0], t[1], va[4 * j + 0], va[4 * j + 1], se, so);
                    fma_pair(t[2], t[3], va[4 * j + 2], va[4 * j + 3], se, so);
                    fma_pair(t[4], t[5], vb[4 * j + 0], vb[4 * j + 1], se, so);
                    fma_pair(t[6], t[7], vb[4 * j + 2], vb[4 * j + 3], se, so);
                }
            }
        } else {
            float v[kF];
#pragma unroll
            for (int c = 0; c < kF / 16; ++c)
                tc_ld16(taddr + col_b + kF * g + 16 * c, *reinterpret_cast<float(*)[16]>(v + 16 * c));
            tc_wait_ld();
            const float4 *sp = reinterpret_cast<const float4 *>(sq + kF * g);
#pragma unroll
            for (int q4 = 0; q4 < kF / 4; ++q4) {
                const float4 s4 = sp[q4];  // the same address in every lane: a broadcast
                float *t = total + kF * g + 4 * q4;
                fma_pair(t[0], t[1], v[4 * q4 + 0], v[4 * q4 + 1], s4.x, s4.y);
                fma_pair(t[2], t[3], v[4 * q4 + 2], v[4 * q4 + 3], s4.z, s4.w);
            }
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int NTOK, bool kBlock>
__global__ void __launch_bounds__(Tc<NTOK, kBlock>::kThreads, 1) __maxnreg__((Tc<NTOK, kBlock>::kMaxRegs))
    w8a8_gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                        const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                        const __grid_constant__ CUtensorMap tm_a, const W8A8Args a) {
    using C = Tc<NTOK, kBlock>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + C::kStages;
    uint64_t *accf = empty + C::kStages;  // [kAcc] accumulator buffer ready
    uint64_t *acce = accf + C::kAcc;      // [kAcc] accumulator buffer drained
    uint64_t *scal = acce + C::kAcc;      // [kAcc] block scales written
    uint64_t *done = scal + C::kAcc;      // all MMAs complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    float *sbuf = reinterpret_cast<float *>(smem + C::kScaleOff);  // Block128: [kAcc][kSBuf] sa * sw
    float *red = reinterpret_cast<float *>(smem);  // totals [NTOK][kRedStride], in the ring at the end

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // token blocks of NTOK rows (more than one only beyond 256 rows): the
    // blocks of one weight tile are neighbours in the grid, so they run side by
    // side and the tile's weights come from HBM once
    const uint32_t tbs = (a.m + NTOK - 1) / NTOK, tb = blockIdx.x % tbs;
    const uint32_t tile_row0 = (blockIdx.x / tbs) * kTileRows;
    const uint32_t tok0 = tb * NTOK;                                             // first token row
    const uint32_t m_loc = a.m - tok0 < (uint32_t)NTOK ? a.m - tok0 : (uint32_t)NTOK;  // rows of this block
    const uint32_t split = gridDim.y, sidx = blockIdx.y;
    const uint32_t kb0 = (a.kb * sidx) / split, kb1 = (a.kb * (sidx + 1)) / split;
    const uint32_t niter = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < C::kAcc; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], C::kEpi);
            mbar_init(&scal[b], 1);
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
    if (a.early_trigger) grid_dep_launch();

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
    // true when the rows tile_row0 .. tile_row0+127 that exist all belong to that segment
    const bool tile_single = tile_row0 + kTileRows <= seg_end || seg_end == a.n;

    // weight scale of this tile for K block kb (Block128 tiles lie in one segment)
    auto tile_sw = [&](uint32_t kb) -> float {
        return tile_row0 < a.n ? __ldg(tile_scale + (size_t)(tile_lrow0 >> 7) * a.kb + kb) : 0.0f;
    };
    // TMA of one K block of this tile's weights into stage `st`
    const uint64_t pol_w = policy_evict_first();
    auto load_weights = [&](uint32_t it, uint8_t *st, uint64_t *bar) {
        const int32_t kk = (int32_t)((kb0 + it) * 128);
        if (QDL_TC_BIGBOX && tile_single) {  // the whole tile lies in one segment: one box
            tma_load_2d(st, tile_big, kk, (int32_t)tile_lrow0, bar, pol_w);
            return;
        }
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
            tma_load_2d(st + b * kWBox, m, kk, (int32_t)lr, bar, pol_w);
        }
    };
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
            const uint64_t pol_a = policy_evict_last();
            constexpr uint32_t kTx = C::kStage;
            // weights of the first stages before waiting for the previous kernel
            const uint32_t head = niter < (uint32_t)C::kStages ? niter : (uint32_t)C::kStages;
            for (uint32_t it = 0; it < head; ++it) {
                mbar_arrive_expect_tx(&full[it], kTx);
                issued = it + 1;
                if (it == a.debug_skip_iter) continue;  // self-test: this stage never lands
                load_weights(it, smem + it * C::kStage, &full[it]);
            }
            grid_dep_wait();  // activations are written by the previous kernel
            for (uint32_t it = 0; it < head; ++it)
                if (it != a.debug_skip_iter)
                    tma_load_2d(smem + it * C::kStage + kWBytes, &tm_a, (int32_t)((kb0 + it) * 128), (int32_t)tok0,
                                &full[it], pol_a);
            for (uint32_t it = head; it < niter; ++it) {
                const uint32_t slot = it % C::kStages, ph = (it / C::kStages) & 1;
                wait(&empty[slot], ph ^ 1, 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], kTx);
                issued = it + 1;
                if (it == a.debug_skip_iter) continue;
                uint8_t *st = smem + slot * C::kStage;
                load_weights(it, st, &full[slot]);
                tma_load_2d(st + kWBytes, &tm_a, (int32_t)((kb0 + it) * 128), (int32_t)tok0, &full[slot], pol_a);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f8<kTileRows, NTOK>();
            const uint32_t sbase = smem_u32(smem);
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t slot = it % C::kStages, ph = (it / C::kStages) & 1;
                const uint32_t b = kBlock ? it % C::kAcc : 0;
                if (kBlock) wait(&acce[b], ((it / C::kAcc) & 1) ^ 1, 4);
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
    } else if (kBlock && warp == 2) {
        // ------------------------------------------------------------ scale warp
        // sa[token, kb] * sw[tile, kb] of each K block into sbuf[b].  The raw
        // scales of the next kSAhead blocks are in flight (cp.async into the
        // stage ring); lane l covers tokens l, l + 32, ..., lane 0 the weight scale.
        constexpr int kPer = (NTOK + 31) / 32, kD = C::kSAhead;
        float *stage = reinterpret_cast<float *>(smem + C::kStageOff);
        grid_dep_wait();  // activation scales come from the previous kernel
        auto issue = [&](uint32_t it) {  // copies of block it into stage slot it % kD
            if (it < niter) {
                float *dst = stage + (it % kD) * C::kSStage;
                const uint32_t kb = kb0 + it;
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const uint32_t tok = 32 * j + lane;
                    if (tok < m_loc) cp_async4(dst + tok, a.sa + (size_t)(tok0 + tok) * a.kb + kb);
                }
                if (lane == 0 && tile_row0 < a.n)
                    cp_async4(dst + NTOK, tile_scale + (size_t)(tile_lrow0 >> 7) * a.kb + kb);
            }
            cp_async_commit();  // one group per block, empty past the end
        };
#pragma unroll
        for (int d = 0; d < kD; ++d) issue((uint32_t)d);
        for (uint32_t it = 0; it < niter; ++it) {
            const uint32_t b = it % C::kAcc;
            cp_async_wait<kD - 1>();  // this lane's copies of block it have landed
            __syncwarp();             // ... and every lane's
            const float *src = stage + (it % kD) * C::kSStage;
            const float sw = tile_row0 < a.n ? src[NTOK] : 0.0f;
            float cur[kPer];
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const uint32_t tok = 32 * j + lane;
                cur[j] = tok < m_loc ? src[tok] * sw : 0.0f;
            }
            __syncwarp();  // the slot is read before it is refilled
            issue(it + kD);
            wait(&acce[b], ((it / C::kAcc) & 1) ^ 1, 64);  // the epilogue is done with sbuf[b]
#pragma unroll
            for (int j = 0; j < kPer; ++j)
                if (32 * j + lane < (uint32_t)NTOK)
                    sbuf[b * C::kSBuf + scale_slot<NTOK>(32 * j + lane)] = cur[j];
            __syncwarp();
            if (lane == 0) mbar_arrive(&scal[b]);
        }
        cp_async_wait<0>();  // no copy in flight when the CTA leaves
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - C::kEpiBase;
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        const int cgrp = e >> 2;    // column group
        const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
        grid_dep_wait();  // activation scales come from the previous kernel
        if constexpr (kBlock) {
            const uint32_t sq = scale_row<NTOK>(cgrp, lane);
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t b = it % C::kAcc;
                wait(&scal[b], (it / C::kAcc) & 1, 32);  // sa * sw of this block
                wait(&accf[b], (it / C::kAcc) & 1, 16);
                tc_fence_after();
                fold_block<NTOK>(taddr, b * NTOK + cgrp * kCpt, sbuf + b * C::kSBuf + sq, total);
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
    if (!a.early_trigger) grid_dep_launch();  // the next kernel may start streaming its weights
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t first = issued > (uint32_t)C::kStages ? issued - C::kStages : 0;
            for (uint32_t it = first; it < issued; ++it)
                if (it != a.debug_skip_iter)
                    mbar_wait(&full[it % C::kStages], (it / C::kStages) & 1, a.wait_limit_ns);
        }
        if (warp == 1 && lane == 0) mbar_wait(done, 0, a.wait_limit_ns);
        __syncthreads();
    }
    grid_dep_wait();  // outputs may be read or written by earlier kernels

    // split-K ranks add into the zeroed f32 output (red.global.add.f32)
    // instead of meeting in the cluster reduction
    const bool add_out = a.accumulate && split > 1;
    // (tok: token row within this block)
    auto add = [&](uint32_t tok, uint32_t r, float v) {
        if (tok < m_loc && r < a.n) atomicAdd(reinterpret_cast<float *>(a.out) + (size_t)(tok0 + tok) * a.ldc + r, v);
    };
    auto store = [&](uint32_t tok, uint32_t r, float v) {  // the single writer of (tok, r)
        if (tok < m_loc && r < a.n) {
            const size_t o = (size_t)(tok0 + tok) * a.ldc + r;
            if (a.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(a.out)[o] = __float2bfloat16_rn(v);
            else if (a.accumulate)
                reinterpret_cast<float *>(a.out)[o] += v;
            else
                reinterpret_cast<float *>(a.out)[o] = v;
        }
    };

    // four consecutive outputs (tok, r .. r+3) of this token block, as one
    // 16-byte store or reduction (8 bytes for bf16) where out is aligned for it
    const uint32_t elt = a.out_bf16 ? 2u : 4u;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(a.out) | ((uintptr_t)a.ldc * elt)) & (4 * elt - 1)) == 0;
    auto put4 = [&](uint32_t tok, uint32_t r, float4 v) {
        if (vec4 && tok < m_loc && r + 4 <= a.n) {
            const size_t o = (size_t)(tok0 + tok) * a.ldc + r;
            float *of = reinterpret_cast<float *>(a.out) + o;
            if (a.out_bf16) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t *>(&lo);
                u.y = *reinterpret_cast<const uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + o) = u;
            } else if (add_out) {
                red_add_v4(of, v);
            } else if (a.accumulate) {
                float4 w = *reinterpret_cast<const float4 *>(of);
                w.x += v.x; w.y += v.y; w.z += v.z; w.w += v.w;
                *reinterpret_cast<float4 *>(of) = w;
            } else {
                *reinterpret_cast<float4 *>(of) = v;
            }
            return;
        }
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (add_out)
                add(tok, r + i, f[i]);
            else
                store(tok, r + i, f[i]);
        }
    };

    // ---------------------------------------------------------------- output
    // Block128: every epilogue thread writes its totals to red[token][row] in
    // the freed stage ring; then the epilogue warps write the block's outputs
    // in 16-byte pieces, or (split > 1 without f32 reductions) the cluster
    // reduction below reads them.  PerRow: each thread owns one row.
    if (warp >= C::kEpiBase) {
        const int e = warp - C::kEpiBase;
        const int quad = warp & 3;
        const int cgrp = e >> 2;
        const uint32_t lrow = 32 * quad + lane;
        const uint32_t row = tile_row0 + lrow;
        if constexpr (kBlock) {
#pragma unroll
            for (int j = 0; j < kCpt; ++j) {
                const uint32_t tok = cgrp * kCpt + frag_tok<C::kFrag>(j, lane);
                const uint32_t jrow = 32 * quad + frag_row<C::kFrag>(j, lane);
                red[tok * kRedStride + jrow] = total[j];
            }
            if (split == 1 || add_out) {
                // every epilogue warp's totals are in place
                asm volatile("bar.sync 1, %0;" ::"r"(C::kEpi * 32) : "memory");
                constexpr uint32_t kR4 = kTileRows / 4;
                for (uint32_t idx = (uint32_t)e * 32 + lane; idx < m_loc * kR4; idx += C::kEpi * 32) {
                    const uint32_t tok = idx / kR4, r4 = idx % kR4;
                    put4(tok, tile_row0 + 4 * r4, *reinterpret_cast<const float4 *>(red + tok * kRedStride + 4 * r4));
                }
            }
            (void)row;
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
                    const float s = tok < m_loc ? ld_dep(a.sa + tok0 + tok) * swr : 0.0f;
                    if (split == 1)
                        store(tok, row, v[i] * s);
                    else if (add_out)
                        add(tok, row, v[i] * s);
                    else
                        red[tok * kRedStride + lrow] = v[i] * s;
                }
            }
            (void)e;
            (void)cgrp;
        }
    }

    if (split > 1 && !add_out) {
        // rank r adds the 4-row chunks 32r/split .. 32(r+1)/split - 1 of every
        // rank's totals, in rank order, and writes them in 16-byte pieces
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        constexpr uint32_t kR4 = kTileRows / 4;
        const uint32_t c_lo = (kR4 * sidx) / split, c_hi = (kR4 * (sidx + 1)) / split;
        const uint32_t span = c_hi - c_lo;
        const float *peer[8];
#pragma unroll
        for (int rk = 0; rk < 8; ++rk) peer[rk] = cluster.map_shared_rank(red, rk < (int)split ? rk : 0);
        for (uint32_t idx = threadIdx.x; idx < span * m_loc; idx += blockDim.x) {
            const uint32_t tok = idx / span, r4 = c_lo + idx % span;
            float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) {  // rank order
                if (rk < (int)split) {
                    const float4 v = *reinterpret_cast<const float4 *>(peer[rk] + tok * kRedStride + 4 * r4);
                    sum.x += v.x;
                    sum.y += v.y;
                    sum.z += v.z;
                    sum.w += v.w;
                }
            }
            put4(tok, tile_row0 + 4 * r4, sum);
        }
        cluster.sync();  // no rank leaves while others still read its totals
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

// ---------------------------------------------------------------- stream-K variant
//
// Block128, f32 output that the caller has zeroed (accumulate mode).  The work
// is the sequence of (tile, K block) units, tile-major; CTA c of P takes units
// [c U / P, (c+1) U / P) and streams them through one ring without stopping at
// tile boundaries, so every CTA moves the same number of weight bytes and no
// CTA waits for a second wave.  The epilogue keeps register totals for the
// current tile; when the CTA's range leaves that tile it stores them if the
// CTA covered the whole tile, and otherwise adds them into the output with f32
// atomics (a tile shared by two or more CTAs).  Roles, barriers and bounded waits are those
// of w8a8_gemm_tc_kernel<NTOK, true>.
template <int NTOK>
__global__ void __launch_bounds__(Tc<NTOK, true>::kThreads, 1) __maxnreg__((Tc<NTOK, true>::kMaxRegs))
    w8a8_streamk_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                        const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                        const __grid_constant__ CUtensorMap tm_a, const W8A8Args a) {
    using C = Tc<NTOK, true>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + C::kStages;
    uint64_t *accf = empty + C::kStages;
    uint64_t *acce = accf + C::kAcc;
    uint64_t *scal = acce + C::kAcc;
    uint64_t *done = scal + C::kAcc;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    float *sbuf = reinterpret_cast<float *>(smem + C::kScaleOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tiles = (a.n + kTileRows - 1) / kTileRows;
    const uint64_t units = (uint64_t)tiles * a.kb;
    const uint32_t u0 = (uint32_t)(units * blockIdx.x / gridDim.x);
    const uint32_t u1 = (uint32_t)(units * (blockIdx.x + 1) / gridDim.x);
    const uint32_t niter = u1 - u0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < C::kAcc; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], C::kEpi);
            mbar_init(&scal[b], 1);
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

    // segment of a tile (Block128 tiles never straddle segments)
    struct TileSeg {
        const float *scale;
        const CUtensorMap *big;
        uint32_t lrow0;
        bool single;
    };
    auto tile_seg = [&](uint32_t tile) {
        const uint32_t r0 = tile * kTileRows;
        TileSeg t;
        uint32_t seg_end;
        if (r0 < a.n1) {
            t.scale = a.sw0; t.lrow0 = r0; t.big = &tm_b0; seg_end = a.n1;
        } else if (r0 < a.n2) {
            t.scale = a.sw1; t.lrow0 = r0 - a.n1; t.big = &tm_b1; seg_end = a.n2;
        } else {
            t.scale = a.sw2; t.lrow0 = r0 - a.n2; t.big = &tm_b2; seg_end = a.n;
        }
        t.single = r0 + kTileRows <= seg_end || seg_end == a.n;
        return t;
    };

    uint32_t issued = 0;
    constexpr int kCpt = C::kCpt;
    float total[kCpt];
#pragma unroll
    for (int j = 0; j < kCpt; ++j) total[j] = 0.0f;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_a);
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            auto load_weights = [&](uint32_t u, uint8_t *st, uint64_t *bar) {
                const uint32_t tile = u / a.kb, kb = u % a.kb;
                const TileSeg t = tile_seg(tile);
                const int32_t kk = (int32_t)(kb * 128);
                if (QDL_TC_BIGBOX && t.single) {
                    tma_load_2d(st, t.big, kk, (int32_t)t.lrow0, bar, pol_w);
                    return;
                }
#pragma unroll 1
                for (int b = 0; b < kTileRows / 16; ++b) {
                    const uint32_t r0 = tile * kTileRows + 16 * b;
                    const CUtensorMap *m;
                    uint32_t lr;
                    if (r0 < a.n1) {
                        m = &tm_w0; lr = r0;
                    } else if (r0 < a.n2) {
                        m = &tm_w1; lr = r0 - a.n1;
                    } else {
                        m = &tm_w2; lr = r0 - a.n2;
                    }
                    tma_load_2d(st + b * kWBox, m, kk, (int32_t)lr, bar, pol_w);
                }
            };
            constexpr uint32_t kTx = C::kStage;
            const uint32_t head = niter < (uint32_t)C::kStages ? niter : (uint32_t)C::kStages;
            for (uint32_t it = 0; it < head; ++it) {
                mbar_arrive_expect_tx(&full[it], kTx);
                issued = it + 1;
                load_weights(u0 + it, smem + it * C::kStage, &full[it]);
            }
            grid_dep_wait();  // activations are written by the previous kernel
            for (uint32_t it = 0; it < head; ++it)
                tma_load_2d(smem + it * C::kStage + kWBytes, &tm_a, (int32_t)(((u0 + it) % a.kb) * 128), 0, &full[it],
                            pol_a);
            for (uint32_t it = head; it < niter; ++it) {
                const uint32_t slot = it % C::kStages, ph = (it / C::kStages) & 1;
                wait(&empty[slot], ph ^ 1, 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], kTx);
                issued = it + 1;
                uint8_t *st = smem + slot * C::kStage;
                load_weights(u0 + it, st, &full[slot]);
                tma_load_2d(st + kWBytes, &tm_a, (int32_t)(((u0 + it) % a.kb) * 128), 0, &full[slot], pol_a);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f8<kTileRows, NTOK>();
            const uint32_t sbase = smem_u32(smem);
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t slot = it % C::kStages, ph = (it / C::kStages) & 1;
                const uint32_t b = it % C::kAcc;
                wait(&acce[b], ((it / C::kAcc) & 1) ^ 1, 4);
                wait(&full[slot], ph, 8);
                if (*abort_flag) break;
                tc_fence_after();
                const uint64_t ad = sw128_desc(sbase + slot * C::kStage);
                const uint64_t bd = sw128_desc(sbase + slot * C::kStage + kWBytes);
                const uint32_t d = tmem + b * NTOK;
#pragma unroll
                for (int k = 0; k < 4; ++k) tc_mma(d, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                tc_commit(&empty[slot]);
                tc_commit(&accf[b]);
            }
            tc_commit(done);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ scale warp
        // as in w8a8_gemm_tc_kernel: the raw scales of the next kSAhead units
        // are in flight in the stage ring
        constexpr int kPer = (NTOK + 31) / 32, kD = C::kSAhead;
        float *stage = reinterpret_cast<float *>(smem + C::kStageOff);
        grid_dep_wait();
        auto issue = [&](uint32_t it) {  // copies of unit u0 + it into stage slot it % kD
            if (it < niter) {
                float *dst = stage + (it % kD) * C::kSStage;
                const uint32_t u = u0 + it, kb = u % a.kb;
#pragma unroll
                for (int j = 0; j < kPer; ++j) {
                    const uint32_t tok = 32 * j + lane;
                    if (tok < a.m && tok < (uint32_t)NTOK) cp_async4(dst + tok, a.sa + (size_t)tok * a.kb + kb);
                }
                if (lane == 0) {
                    const TileSeg t = tile_seg(u / a.kb);
                    cp_async4(dst + NTOK, t.scale + (size_t)(t.lrow0 >> 7) * a.kb + kb);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int d = 0; d < kD; ++d) issue((uint32_t)d);
        for (uint32_t it = 0; it < niter; ++it) {
            const uint32_t b = it % C::kAcc;
            cp_async_wait<kD - 1>();
            __syncwarp();
            const float *src = stage + (it % kD) * C::kSStage;
            const float sw = src[NTOK];
            float cur[kPer];
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const uint32_t tok = 32 * j + lane;
                cur[j] = tok < a.m && tok < (uint32_t)NTOK ? src[tok] * sw : 0.0f;
            }
            __syncwarp();
            issue(it + kD);
            wait(&acce[b], ((it / C::kAcc) & 1) ^ 1, 64);
#pragma unroll
            for (int j = 0; j < kPer; ++j)
                if (32 * j + lane < (uint32_t)NTOK)
                    sbuf[b * C::kSBuf + scale_slot<NTOK>(32 * j + lane)] = cur[j];
            __syncwarp();
            if (lane == 0) mbar_arrive(&scal[b]);
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - C::kEpiBase;
        const int quad = warp & 3;
        const int cgrp = e >> 2;
        const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
        const uint32_t sq = scale_row<NTOK>(cgrp, lane);
        grid_dep_wait();  // scales come from, and the output is shared with, earlier kernels
        for (uint32_t it = 0; it < niter; ++it) {
            const uint32_t b = it % C::kAcc;
            wait(&scal[b], (it / C::kAcc) & 1, 32);
            wait(&accf[b], (it / C::kAcc) & 1, 16);
            tc_fence_after();
            fold_block<NTOK>(taddr, b * NTOK + cgrp * kCpt, sbuf + b * C::kSBuf + sq, total);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
            // the range leaves this tile: a tile this CTA covers whole is
            // stored, the part of a tile shared with a neighbour is added
            const uint32_t u = u0 + it;
            if (it + 1 == niter || (u + 1) % a.kb == 0) {
                const uint32_t tile = u / a.kb;
                const bool whole = tile * a.kb >= u0 && (tile + 1) * a.kb <= u1;
                if (!*abort_flag) {
                    // this thread's first output (total 0) and how many tokens
                    // and rows from it exist; total j lies frag_tok(j) - frag_tok(0)
                    // tokens and frag_row(j) - frag_row(0) rows further on
                    const uint32_t tok0 = cgrp * kCpt + frag_tok<C::kFrag>(0, lane);
                    const uint32_t row0 = tile * kTileRows + 32 * quad + frag_row<C::kFrag>(0, lane);
                    const int nt = (int)a.m - (int)tok0, nr = (int)a.n - (int)row0;
                    float *o0 = reinterpret_cast<float *>(a.out) + (size_t)tok0 * a.ldc + row0;
                    // a tile this CTA covers whole over a zeroed output is stored; any
                    // other (shared, or QDL_OUT_F32_ADD) is added with reductions, which
                    // for a single writer is one exact add per element
                    if (whole && a.out_zeroed) {
#pragma unroll
                        for (int j = 0; j < kCpt; ++j) {
                            const int dt = (int)(frag_tok<C::kFrag>(j, lane) - frag_tok<C::kFrag>(0, lane));
                            const int dr = (int)(frag_row<C::kFrag>(j, lane) - frag_row<C::kFrag>(0, lane));
                            if (dt < nt && dr < nr) o0[(size_t)dt * a.ldc + dr] = total[j];
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kCpt; ++j) {
                            const int dt = (int)(frag_tok<C::kFrag>(j, lane) - frag_tok<C::kFrag>(0, lane));
                            const int dr = (int)(frag_row<C::kFrag>(j, lane) - frag_row<C::kFrag>(0, lane));
                            if (dt < nt && dr < nr) atomicAdd(o0 + (size_t)dt * a.ldc + dr, total[j]);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < kCpt; ++j) total[j] = 0.0f;
            }
        }
    }

    // ---------------------------------------------------------------- drain after a timeout
    __syncthreads();
    grid_dep_launch();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t first = issued > (uint32_t)C::kStages ? issued - C::kStages : 0;
            for (uint32_t it = first; it < issued; ++it)
                mbar_wait(&full[it % C::kStages], (it / C::kStages) & 1, a.wait_limit_ns);
        }
        if (warp == 1 && lane == 0) mbar_wait(done, 0, a.wait_limit_ns);
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

// Cluster reduction of one split CTA, in K-block units: its partials grow
// with the token count (measured: one K block of time per 4 tokens).
// Where split-K ranks add into a zeroed output with f32 reductions instead,
// the 256-token ranks cost about 4 blocks: split 2 took the 256-row gate/up
// GEMV from 123.8 to 103.7 us (1.47 waves of 224 tiles become 2.95).
constexpr double tc_reduce_cost(int ntok, bool accumulate) {
    return accumulate && ntok >= 256 ? 4.0 : ntok / 4.0;
}

template <int NTOK, bool kBlock>
const uint32_t *cta_slots_tc() {
    using C = Tc<NTOK, kBlock>;
    static std::mutex mu;
    static std::vector<std::vector<uint32_t>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    if (cache[dev].empty()) {
        const void *f = (const void *)w8a8_gemm_tc_kernel<NTOK, kBlock>;
        cudaFuncSetAttribute(w8a8_gemm_tc_kernel<NTOK, kBlock>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kAlloc);
        cache[dev].assign(8, 0);
        resident_cta_slots(f, C::kThreads, C::kAlloc, resident_ctas(f, C::kThreads, C::kAlloc, C::kTmemCols),
                           cache[dev].data());
    }
    return cache[dev].data();
}

template <int NTOK, bool kBlock>
cudaError_t launch_tc_variant(const W8A8Args &a, const CUtensorMap (&maps)[7], cudaStream_t s) {
    using C = Tc<NTOK, kBlock>;
    // output tiles x token blocks (more than one block only beyond 256 rows)
    const uint32_t tiles = (a.n + kTileRows - 1) / kTileRows * ((a.m + NTOK - 1) / NTOK);
    const uint32_t split = choose_split_k(tiles, a.kb, cta_slots_tc<NTOK, kBlock>(), tc_reduce_cost(NTOK, a.accumulate != 0));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, split, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kAlloc;
    cfg.stream = s;
    // Split-K ranks that add into a zeroed output never meet.  When the
    // previous call releases this one early, launching them without a cluster
    // lets each CTA take a slot as soon as one frees instead of waiting for
    // `split` free slots in one GPC: 7.58 -> 7.21 us per call on the 25 MB QKV
    // projection at M=8.  Without the early release, clusters measured faster
    // (1 MB per-row projection at M=1: 4.44 us clustered, 4.81 without).
    const bool clustered = split > 1 && !(a.accumulate && a.early_trigger && QDL_TC_ADD_NOCLUSTER);
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (clustered) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = split;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (QDL_TUNE_PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, w8a8_gemm_tc_kernel<NTOK, kBlock>, maps[0], maps[1], maps[2], maps[3],
                              maps[4], maps[5], maps[6], a);
}

template <int NTOK, bool kBlock>
void plan_tc_variant(const W8A8Args &a, PlanInfo *p) {
    using C = Tc<NTOK, kBlock>;
    const uint32_t *slots = cta_slots_tc<NTOK, kBlock>();
    p->kernel = 0;
    p->mma_n = NTOK;
    p->tiles = (a.n + kTileRows - 1) / kTileRows;
    p->split = choose_split_k(p->tiles * ((a.m + NTOK - 1) / NTOK), a.kb, slots, tc_reduce_cost(NTOK, a.accumulate != 0));
    p->stages = C::kStages;
    p->threads = C::kThreads;
    p->smem = C::kAlloc;
    p->clusters = (int)(slots[p->split - 1] / p->split);
}

template <bool kBlock>
void plan_tc_rows(const W8A8Args &a, uint32_t ntok, PlanInfo *p) {
    switch (ntok) {
        case 16: return plan_tc_variant<16, kBlock>(a, p);
        case 32: return plan_tc_variant<32, kBlock>(a, p);
        case 64: return plan_tc_variant<64, kBlock>(a, p);
        case 128: return plan_tc_variant<128, kBlock>(a, p);
        default: return plan_tc_variant<256, kBlock>(a, p);
    }
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

// Stream-K: one CTA per resident slot (the same shared memory and threads as
// the split-K Block128 variant, no cluster), at most one unit each.
template <int NTOK>
cudaError_t launch_streamk_variant(const W8A8Args &a, const CUtensorMap (&maps)[7], cudaStream_t s) {
    using C = Tc<NTOK, true>;
    static std::mutex mu;
    static std::vector<uint32_t> slots;  // per device
    int dev = 0;
    cudaGetDevice(&dev);
    uint32_t p;
    {
        std::lock_guard<std::mutex> lock(mu);
        if ((int)slots.size() <= dev) slots.resize(dev + 1, 0);
        if (slots[dev] == 0) {
            const void *f = (const void *)w8a8_streamk_kernel<NTOK>;
            cudaFuncSetAttribute(w8a8_streamk_kernel<NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kAlloc);
            slots[dev] = (uint32_t)(resident_ctas(f, C::kThreads, C::kAlloc, C::kTmemCols) * device_sm_count());
        }
        p = slots[dev];
    }
    const uint64_t units = (uint64_t)((a.n + kTileRows - 1) / kTileRows) * a.kb;
    if (units < p) p = (uint32_t)units;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, w8a8_streamk_kernel<NTOK>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                              maps[6], a);
}

cudaError_t launch_streamk_rows(const W8A8Args &a, const CUtensorMap (&maps)[7], uint32_t ntok, cudaStream_t s) {
    static_assert(QDL_STREAMK_MIN_NTOK >= 16 && QDL_STREAMK_MAX_NTOK <= 128, "stream-K is instantiated for 16..128");
    switch (ntok) {
        case 16: return launch_streamk_variant<16>(a, maps, s);
        case 32: return launch_streamk_variant<32>(a, maps, s);
        case 64: return launch_streamk_variant<64>(a, maps, s);
        default: return launch_streamk_variant<128>(a, maps, s);
    }
}

cudaError_t weight_maps(const W8A8Args &a, const uint8_t *const seg_w[3], const uint32_t seg_n[3],
                        CUtensorMap (&maps)[7]) {
    for (int i = 0; i < 3; ++i) {  // 16-row boxes x3, 128-row boxes x3
        cudaError_t e = make_tmap_u8(&maps[i], seg_w[i], a.k, seg_n[i], a.k, 128, 16);
        if (e != cudaSuccess) return e;
        e = make_tmap_u8(&maps[3 + i], seg_w[i], a.k, seg_n[i], a.k, 128, kTileRows);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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
    cudaError_t e = weight_maps(a, seg_w, seg_n, maps);
    if (e != cudaSuccess) return e;
    const uint32_t ntok = tc_bucket(a.m);
    e = make_tmap_u8(&maps[6], a.q, a.k, a.m, a.k, 128, ntok < 256 ? ntok : 256);
    if (e != cudaSuccess) return e;
    if (a.accumulate && w8a8_streamk_applies(format, a.m)) return launch_streamk_rows(a, maps, ntok, s);
    W8A8Args b = a;
    b.early_trigger = ntok <= QDL_TC_EARLY_MAX_NTOK && (uint64_t)a.n * a.k >= QDL_TC_EARLY_TRIGGER_BYTES ? 1u : 0u;
    return format == QDL_SCALE_BLOCK128 ? launch_tc_rows<true>(b, maps, ntok, s) : launch_tc_rows<false>(b, maps, ntok, s);
}

bool w8a8_streamk_applies(int format, uint32_t rows) {
    const uint32_t ntok = tc_bucket(rows);
    return format == QDL_SCALE_BLOCK128 && ntok >= QDL_STREAMK_MIN_NTOK && ntok <= QDL_STREAMK_MAX_NTOK;
}

cudaError_t plan_w8a8_gemm_tc(const W8A8Args &a, int format, PlanInfo *p) {
    const uint32_t ntok = tc_bucket(a.m);
    if (format == QDL_SCALE_BLOCK128)
        plan_tc_rows<true>(a, ntok, p);
    else
        plan_tc_rows<false>(a, ntok, p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_tc_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_tc_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_tc_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
