// AWQ INT4 fused Q/K/V projection on the 5th-generation tensor cores
// (fused_int4_qkv.rs: fused_int4_qkv_q, fused_int4_qkv_k, fused_int4_qkv_v,
// unpack_awq_qkv, QKV_AWQ_SHIFTS).  One launch covers all three projections
// for up to 32 token rows; this path serves group size 128 and projection
// widths that are multiples of 32 (the others take the CUDA-core or the
// mma.sync kernel).
//
// Arithmetic.  x~ is x rounded to f16 (the only approximation,
// |x~ - x| <= 2^-11 |x|).  A packed word holds the nibbles of 8 columns in the
// AWQ order: physical nibble p (bits 4p..4p+3) is column {0,2,4,6,1,3,5,7}[p].
// OR-ing a masked nibble pair into the f16 pattern of 1024 (0x6400) gives the
// exact f16 pair (1024 + nib, 1024 + nib').  The tensor core accumulates
// acc = sum_k x~ (1024 + nib) in f32, and per group g the epilogue adds
//   s acc - s (1024 + z) sum_k x~  =  s sum_k x~ (nib - z)
// (exact algebra; the large 1024 terms cancel with f32 rounding far below the
// tolerance).
//
// Work.  The (128-column tile, 128-K unit) pairs of all three projections,
// tile-major (a unit is one quantisation group), are cut into one contiguous
// range per CTA (stream-K, one CTA per SM), so every SM streams the same
// number of code bytes in one wave.  The caller's outputs are zeroed first
// (int4_zero_kernel) and each CTA adds its per-tile totals with f32 atomics
// when its range leaves a tile.
//
// The A operand (weights as f16, M = 128 columns x K = 128 per unit) lives in
// tensor memory: one 64-column slot per unit, written by the converters with
// tcgen05.st, so neither a shared-memory round trip nor a proxy fence sits
// between the code stream and the MMAs.  Tensor-memory lane L holds column
// 32 (L / 32) + 8 ((L % 32) / 8) + {0,2,4,6,1,3,5,7}[L % 8] of the tile (the
// order the nibble transpose leaves them in); the accumulator rows follow the
// same order.
//
// Roles (one CTA):
//   warp 0, one lane : TMA producer: per unit the [128 K x 16 words] codes and
//                      the group's 128 scales and zeros, into a ring; it
//                      starts before the programmatic-launch wait (weights
//                      do not come from the previous kernel) and skips the
//                      prologue.
//   prologue, others : after that wait, x of every unit of the range -> x~ in
//                      the f16 B operand layout (K-major, 128-byte swizzle,
//                      two 64-K atoms per unit) and sum x~ per unit and token.
//   warps 1, 2       : MMA issuers for even and odd units: eight kind::f16
//                      MMAs per unit (M = 128, N = tokens, K = 16, A from
//                      tensor memory) into one of four accumulators.
//   warps 3..10      : two converter groups of four warps (one per tensor
//                      memory lane quarter), for even and odd units: per 8
//                      K rows, one code word per lane and an 8 x 8 nibble
//                      transpose across the lanes of each word column (three
//                      shuffle steps, applied to eight blocks at a time), then
//                      four f16 pairs (k, k + 1) per lane; 32 pairs per lane
//                      go to tensor memory in one tcgen05.st.  Also the fold
//                      coefficients (s, s (1024 + z)) of the unit's group.
//   warps 11..18     : two epilogue sets of four warps, for even and odd
//                      units: tcgen05.ld of the unit's accumulator and two
//                      FMAs per output into register totals; atomic adds at
//                      the end of each tile of the range.
// Every wait is bounded (fault word, drain, return).
#include <cuda_fp16.h>

#include <mutex>
#include <vector>

#include "tma_pipe.cuh"

namespace qdl {

static __device__ uint32_t g_int4_fault;

namespace {

constexpr int kCols = 128;     // output columns per tile (MMA M)
constexpr int kUnitK = 128;    // K rows per unit: one group
constexpr int kGroupK = 128;
constexpr int kGroups = 2;     // converter groups (even / odd units)
constexpr int kSets = 2;       // epilogue sets (even / odd units)
constexpr int kQuarterWarps = 4;
constexpr int kConvBase = 3;
constexpr int kEpiBase = kConvBase + kGroups * kQuarterWarps;
constexpr int kThreadsI4 = (kEpiBase + kSets * kQuarterWarps) * 32;
constexpr uint32_t kCodeBytes = kUnitK * (kCols / 8) * 4;     // 128 rows x 16 words = 8 KB
constexpr uint32_t kStageBytes = kCodeBytes + 2 * kCols * 4;  // + 128 scales + 128 zeros
constexpr int kAcc = 4;        // accumulators
constexpr uint32_t kASlotCols = kUnitK / 2;  // tensor-memory columns of one unit's A (f16 pairs)
constexpr int kSlots = 12;     // fold coefficients of a unit, rewritten after its fold

template <int NTOK>
struct I4 {
    static constexpr int kRing = NTOK <= 16 ? 10 : 8;            // code stages
    static constexpr uint32_t kMaxUnits = NTOK <= 16 ? 12 : 10;  // units per CTA (x~ of all of them is resident)
    static constexpr uint32_t kAccCols = kAcc * NTOK;
    static constexpr int kASlots = (int)((512 - kAccCols) / kASlotCols) & ~1;  // A slots in tensor memory (even)
    static constexpr uint32_t kBAtom = NTOK * 128;                // NTOK rows x 64 k of f16 (one 128-byte swizzle atom)
    static constexpr uint32_t kBOp = 2 * kBAtom;                  // f16 B operand of a unit: two atoms along K
    static constexpr uint32_t kRingOff = 0;
    static constexpr uint32_t kBOff = kRingOff + kRing * kStageBytes;
    static constexpr uint32_t kSxOff = kBOff + kMaxUnits * kBOp;        // [kMaxUnits][NTOK] f32
    static constexpr uint32_t kCoefOff = kSxOff + kMaxUnits * NTOK * 4;  // [kSlots][kCols] float2
    static constexpr uint32_t kBarOff = kCoefOff + kSlots * kCols * 8;
    static constexpr uint32_t kBytes = kBarOff + 1024;  // barriers, the tensor-memory slot and the abort flag
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static_assert(NTOK == 16 || NTOK == 32, "token buckets");
    static_assert(kASlots % 2 == 0 && kAcc % 2 == 0 && kSlots % 2 == 0 && kRing % 2 == 0,
                  "even and odd units never share a barrier");
    static_assert(kASlots + kAcc <= kSlots, "a coefficient slot is rewritten only after its unit is folded");
    static_assert(kBOff % 1024 == 0 && kBAtom % 1024 == 0, "operand alignment");
    static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// K-major operand, 128-byte swizzle: rows of 64 f16 (one atom wide), 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t saddr, uint32_t atom_stride) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(atom_stride >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// kind::f16: D f32, A and B f16, both K-major, M = 128.
template <int NTOK>
__device__ __forceinline__ constexpr uint32_t idesc_f16() {
    return (1u << 4) | ((uint32_t)(NTOK >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D (tensor memory) += A (tensor memory) * B (shared memory descriptor)
__device__ __forceinline__ void mma_f16_ta(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 consecutive tensor-memory columns of this thread's lane <- r[0..31]
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t h2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The published AWQ / Marlin-style interleave-to-f16 conversion, implemented
// from its description: a 4-bit value ORed into the mantissa of the f16
// pattern of 1024.0 (0x6400) is the f16 number 1024 + nib, two per word.
__device__ __forceinline__ uint32_t lop3_mask_or(uint32_t v, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(0x64006400u));  // (v & mask) | 0x64006400
    return r;
}

// One step of the 8 x 8 nibble transpose across the 8 lanes of a word
// column: lanes whose bit d is clear keep their low blocks and take the
// partner's low blocks into their high ones; the others the reverse
// (blocks of 4 d nibbles; m marks the low blocks).
__device__ __forceinline__ uint32_t transpose_step(uint32_t v, uint32_t lane, uint32_t d, uint32_t m) {
    const bool up = (lane & d) != 0;
    const uint32_t s = 4 * d;
    const uint32_t send = __funnelshift_l(v, v, up ? s : 32 - s);  // rotation: the stray blocks are masked off
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, d);
    const uint32_t take = up ? m : ~m;  // bits taken from the partner
    return (v & ~take) | (recv & take);
}

// Zero the three outputs [m, n] before the stream-K GEMV adds into them.
__global__ void __launch_bounds__(256) int4_zero_kernel(const Int4Args a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the GEMV starts streaming codes now
    asm volatile("griddepcontrol.wait;" ::: "memory");               // earlier kernels may still use the outputs
    const size_t nq = (size_t)a.m * a.nq, nkv = (size_t)a.m * a.nkv;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nq + 2 * nkv; i += stride) {
        if (i < nq)
            a.out0[i] = 0.0f;
        else if (i < nq + nkv)
            a.out1[i - nq] = 0.0f;
        else
            a.out2[i - nq - nkv] = 0.0f;
    }
}

template <int NTOK>
__global__ void __launch_bounds__(kThreadsI4, 1)
    int4_qkv_tc_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                       const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_s0,
                       const __grid_constant__ CUtensorMap tm_s1, const __grid_constant__ CUtensorMap tm_s2,
                       const __grid_constant__ CUtensorMap tm_z0, const __grid_constant__ CUtensorMap tm_z1,
                       const __grid_constant__ CUtensorMap tm_z2, const Int4Args a) {
    using C = I4<NTOK>;
    constexpr int kRing = C::kRing;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);  // [kRing] codes, scales, zeros landed
    uint64_t *empty = full + kRing;                                     // [kRing] unit converted
    uint64_t *opfull = empty + kRing;                                   // [kASlots] A slot written
    uint64_t *opempty = opfull + C::kASlots;                            // [kASlots] A slot consumed by the MMAs
    uint64_t *accf = opempty + C::kASlots;                              // [kAcc] unit accumulated
    uint64_t *acce = accf + kAcc;                                       // [kAcc] unit folded
    uint64_t *cfull = acce + kAcc;                                      // [kSlots] fold coefficients written
    uint64_t *done = cfull + kSlots;                                    // [2] every MMA of an issuer complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 2);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    uint8_t *bop = smem + C::kBOff;                                     // [kMaxUnits][NTOK rows x 128 B]
    float *sxall = reinterpret_cast<float *>(smem + C::kSxOff);        // [kMaxUnits][NTOK]
    float2 *coef = reinterpret_cast<float2 *>(smem + C::kCoefOff);     // [kSlots][kCols]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t upt = a.k / kUnitK;  // units per tile
    const uint64_t all_units = (uint64_t)(a.tiles_q + 2 * a.tiles_kv) * upt;
    const uint32_t v0 = (uint32_t)(all_units * blockIdx.x / gridDim.x);
    const uint32_t nunits = (uint32_t)(all_units * (blockIdx.x + 1) / gridDim.x) - v0;  // 1..kMaxUnits (host)

    // projection of a column tile: codes, scales, zeros, output, width and first column
    struct Tile {
        const CUtensorMap *w, *s, *z;
        float *out;
        uint32_t n, col0;
    };
    auto tile_of = [&](uint32_t tile) {
        Tile t;
        if (tile < a.tiles_q) {
            t.w = &tm_w0; t.s = &tm_s0; t.z = &tm_z0; t.out = a.out0; t.n = a.nq;
        } else if (tile < a.tiles_q + a.tiles_kv) {
            tile -= a.tiles_q;
            t.w = &tm_w1; t.s = &tm_s1; t.z = &tm_z1; t.out = a.out1; t.n = a.nkv;
        } else {
            tile -= a.tiles_q + a.tiles_kv;
            t.w = &tm_w2; t.s = &tm_s2; t.z = &tm_z2; t.out = a.out2; t.n = a.nkv;
        }
        t.col0 = tile * kCols;
        return t;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kQuarterWarps);
        }
        for (int i = 0; i < C::kASlots; ++i) {
            mbar_init(&opfull[i], kQuarterWarps);
            mbar_init(&opempty[i], 1);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], kQuarterWarps);
        }
        for (int i = 0; i < kSlots; ++i) mbar_init(&cfull[i], kQuarterWarps);
        mbar_init(&done[0], 1);
        mbar_init(&done[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fault = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(&g_int4_fault, code);
    };
    // ready phases return at once; the abort flag is read only on the slow path
    auto wait = [&](uint64_t *bar, uint32_t parity, uint32_t code) {
        if (mbar_try_wait(bar, parity)) return;
        if (!*abort_flag && !mbar_wait(bar, parity, kWaitLimitNs)) fault(code);
    };

    // ---------------------------------------------------------------- code stream (before the dependency wait)
    uint32_t codes_issued = 0;
    uint64_t pol_w = 0;
    // lanes 0, 1, 2 of the producer warp issue a unit's codes, scales and
    // zeros together (one issuing thread takes about 100 ns per copy); lane 0
    // also posts the transaction count, which may follow the other lanes'
    // copies (the phase cannot complete before lane 0 arrives)
    auto load_codes = [&](uint32_t u) {
        const uint32_t slot = u % kRing, v = v0 + u, ku = v % upt;
        const Tile t = tile_of(v / upt);
        uint8_t *st = smem + slot * kStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[slot], kStageBytes);
            tma_load_2d(st, t.w, (int32_t)(t.col0 / 8), (int32_t)(ku * kUnitK), &full[slot], pol_w);
        } else if (lane == 1) {
            tma_load_2d(st + kCodeBytes, t.s, (int32_t)t.col0, (int32_t)ku, &full[slot], pol_w);
        } else {
            tma_load_2d(st + kCodeBytes + kCols * 4, t.z, (int32_t)t.col0, (int32_t)ku, &full[slot], pol_w);
        }
        codes_issued = u + 1;
    };
    if (warp == 0 && lane < 3) {
        // codes, scales and zeros are read once per call; a 256-byte L2 fill
        // serves the neighbouring column tiles, which read the same K rows at
        // about the same time, so no eviction hint
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_w));
        const uint32_t head = nunits < (uint32_t)kRing ? nunits : (uint32_t)kRing;
        for (uint32_t u = 0; u < head; ++u) load_codes(u);
    }

    // ---------------------------------------------------------------- prologue: x~ and sum x~ of every unit
    // (every warp but the producer's, which keeps issuing the code stream)
    if (warp != 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // x (and the zeroed outputs) come from earlier kernels
        const uint32_t m_used = a.m < (uint32_t)NTOK ? a.m : (uint32_t)NTOK;
        const uint32_t items = nunits * NTOK * 16;  // (unit, token, 8-value chunk of 128 k), chunk fastest
        const uint32_t nthr = blockDim.x - 32;      // a multiple of 16
        for (uint32_t i0 = 0; i0 < items; i0 += nthr) {
            const uint32_t i = i0 + threadIdx.x - 32;
            const uint32_t c = i & 15, tok = (i >> 4) % NTOK, u = (i >> 4) / NTOK;
            uint4 h = make_uint4(0, 0, 0, 0);
            float sum = 0.0f;
            if (i < items && tok < m_used) {
                const uint32_t ku = (v0 + u) % upt;
                const float4 *xp = reinterpret_cast<const float4 *>(a.x + (size_t)tok * a.k + ku * kUnitK + 8 * c);
                const float4 p0 = ld_dep(xp), p1 = ld_dep(xp + 1);
                h = make_uint4(h2_bits(p0.x, p0.y), h2_bits(p0.z, p0.w), h2_bits(p1.x, p1.y), h2_bits(p1.z, p1.w));
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&h.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&h.y));
                const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&h.z));
                const float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&h.w));
                sum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            if (i < items) {
                // atom c / 8 (64 k each), 16-byte chunk c % 8 of row tok, 128-byte swizzle
                *reinterpret_cast<uint4 *>(bop + u * C::kBOp + (c >> 3) * C::kBAtom + tok * 128 +
                                           (((c & 7) ^ (tok & 7)) << 4)) = h;
                if (c == 0) sxall[u * NTOK + tok] = sum;
            }
        }
        fence_proxy_async_smem();  // B operands written by threads -> visible to the tensor core
        asm volatile("bar.sync 1, %0;" ::"r"(blockDim.x - 32) : "memory");
    }

    float total[NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) total[t] = 0.0f;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane < 3) {
            // unit s converted: its stage takes unit s + kRing; the three
            // lanes take the same decision (lane 0's view of the abort flag)
            for (uint32_t s = 0; s + kRing < nunits; ++s) {
                wait(&empty[s % kRing], (s / kRing) & 1, 1);
                __syncwarp(0x7u);
                const uint32_t stop = __shfl_sync(0x7u, *abort_flag ? 1u : 0u, 0);
                if (stop) break;
                load_codes(s + kRing);
            }
        }
    } else if (warp <= 2) {
        // ------------------------------------------------------------ MMA issuers (even / odd units)
        if (lane == 0) {
            const uint32_t j = (uint32_t)warp - 1;
            constexpr uint32_t idesc = idesc_f16<NTOK>();
            const uint32_t bbase = smem_u32(bop);
            for (uint32_t u = j; u < nunits; u += 2) {
                const uint32_t sa = u % C::kASlots, b = u % kAcc;
                wait(&acce[b], ((u / kAcc) & 1) ^ 1, 2);
                wait(&opfull[sa], (u / C::kASlots) & 1, 4);
                if (*abort_flag) break;
                fence_after();
                const uint32_t aslot = tmem + C::kAccCols + sa * kASlotCols, bbuf = bbase + u * C::kBOp;
                const uint32_t d = tmem + b * NTOK;
#pragma unroll
                for (int i = 0; i < kUnitK / 16; ++i)  // K = 16 per MMA: 8 columns of A, 32 bytes of a B atom
                    mma_f16_ta(d, aslot + 8 * i, desc_k_sw128(bbuf + (i >> 2) * C::kBAtom + (i & 3) * 32, C::kBAtom),
                               idesc, i > 0 ? 1u : 0u);
                commit(&opempty[sa]);
                commit(&accf[b]);
            }
            commit(&done[j]);
        }
    } else if (warp < kEpiBase) {
        // ------------------------------------------------------------ converter groups (even / odd units)
        const uint32_t g = (uint32_t)(warp - kConvBase) / kQuarterWarps;
        const uint32_t q = (uint32_t)warp & 3;           // tensor-memory lane quarter: tile columns 32 q ..
        const uint32_t i8 = lane & 7, wj = lane >> 3;    // lane in its word column, word column 4 q + wj
        const uint32_t krow = (i8 < 4 ? 2 * i8 : 2 * (i8 - 4) + 1);  // K row (of 8) this lane loads: nibble slots
                                                                     // (r, r + 4) end up holding K rows (2r, 2r + 1)
        const uint32_t col = 32 * q + 8 * wj + (i8 < 4 ? 2 * i8 : 2 * (i8 - 4) + 1);  // column this lane ends with
        const uint32_t taddr = tmem + ((32 * q) << 16) + C::kAccCols;
        for (uint32_t u = g; u < nunits; u += kGroups) {
            const uint32_t slot = u % kRing, sa = u % C::kASlots, cs = u % kSlots;
            wait(&opempty[sa], ((u / C::kASlots) & 1) ^ 1, 16);
            wait(&full[slot], (u / kRing) & 1, 16);
            if (*abort_flag) break;
            const uint8_t *st = smem + slot * kStageBytes;
            // per 8 K rows: one word per lane, transposed so that lane i8 holds
            // nibble i8 (column col) of the 8 rows, then 4 f16 pairs (k, k + 1);
            // eight 8-row blocks at a time, each transpose step over all eight
            // so that their shuffles overlap
#pragma unroll
            for (int half = 0; half < kUnitK / 64; ++half) {
                uint32_t v[8];
#pragma unroll
                for (int blk = 0; blk < 8; ++blk)
                    v[blk] = *reinterpret_cast<const uint32_t *>(st + (64 * half + 8 * blk + krow) * 64 + (4 * q + wj) * 4);
#pragma unroll
                for (int blk = 0; blk < 8; ++blk) v[blk] = transpose_step(v[blk], lane, 4, 0x0000FFFFu);
#pragma unroll
                for (int blk = 0; blk < 8; ++blk) v[blk] = transpose_step(v[blk], lane, 2, 0x00FF00FFu);
#pragma unroll
                for (int blk = 0; blk < 8; ++blk) v[blk] = transpose_step(v[blk], lane, 1, 0x0F0F0F0Fu);
                uint32_t r[32];
#pragma unroll
                for (int blk = 0; blk < 8; ++blk) {
                    r[4 * blk + 0] = lop3_mask_or(v[blk], 0x000F000Fu);
                    r[4 * blk + 1] = lop3_mask_or(v[blk] >> 4, 0x000F000Fu);
                    r[4 * blk + 2] = lop3_mask_or(v[blk] >> 8, 0x000F000Fu);
                    r[4 * blk + 3] = lop3_mask_or(v[blk] >> 12, 0x000F000Fu);
                }
                st32(taddr + sa * kASlotCols + 32 * half, r);
            }
            // fold coefficients of column col: (s, s (1024 + z))
            const float sc = reinterpret_cast<const float *>(st + kCodeBytes)[col];
            const float zr = reinterpret_cast<const float *>(st + kCodeBytes + kCols * 4)[col];
            coef[cs * kCols + 32 * q + lane] = make_float2(sc, sc * (1024.0f + zr));
            wait_st();
            fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[slot]);
                mbar_arrive(&opfull[sa]);
                mbar_arrive(&cfull[cs]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue sets (even / odd units)
        const uint32_t e = (uint32_t)(warp - kEpiBase) / kQuarterWarps;
        const uint32_t q = (uint32_t)warp & 3;  // tensor-memory lane quarter of this warp
        const uint32_t i8 = lane & 7;
        const uint32_t col = 32 * q + 8 * (lane >> 3) + (i8 < 4 ? 2 * i8 : 2 * (i8 - 4) + 1);  // column of lane 32 q + lane
        const uint32_t taddr = tmem + ((32 * q) << 16);
        const uint32_t m_used = a.m < (uint32_t)NTOK ? a.m : (uint32_t)NTOK;
        for (uint32_t u = e; u < nunits; u += kSets) {
            const uint32_t b = u % kAcc, cs = u % kSlots;
            wait(&cfull[cs], (u / kSlots) & 1, 32);
            wait(&accf[b], (u / kAcc) & 1, 32);
            if (*abort_flag) break;
            fence_after();
            float v[NTOK];
#pragma unroll
            for (int c = 0; c < NTOK / 16; ++c)
                ld16(taddr + b * NTOK + 16 * c, *reinterpret_cast<float(*)[16]>(v + 16 * c));
            wait_ld();
            const float2 cf = coef[cs * kCols + 32 * q + lane];
            const float *sx = sxall + u * NTOK;
#pragma unroll
            for (int t = 0; t < NTOK; ++t) total[t] += fmaf(cf.x, v[t], -cf.y * sx[t]);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
            // this set's last unit of the tile in the range: add its totals into the zeroed output
            const uint32_t vu = v0 + u, tile = vu / upt;
            if (u + kSets >= nunits || (vu + kSets) / upt != tile) {
                const Tile t = tile_of(tile);
                if (t.col0 + col < t.n) {
#pragma unroll
                    for (int jt = 0; jt < NTOK; ++jt)
                        if ((uint32_t)jt < m_used) atomicAdd(t.out + (size_t)jt * t.n + t.col0 + col, total[jt]);
                }
#pragma unroll
                for (int jt = 0; jt < NTOK; ++jt) total[jt] = 0.0f;
            }
        }
    }

    // ---------------------------------------------------------------- drain after a timeout
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t c0 = codes_issued > (uint32_t)kRing ? codes_issued - kRing : 0;
            for (uint32_t u = c0; u < codes_issued; ++u) mbar_wait(&full[u % kRing], (u / kRing) & 1, kWaitLimitNs);
        }
        if ((warp == 1 || warp == 2) && lane == 0) mbar_wait(&done[warp - 1], 0, kWaitLimitNs);
        __syncthreads();
    }
    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// ---------------------------------------------------------------- host side

template <int NTOK>
uint32_t cta_slots_i4() {
    static std::mutex mu;
    static std::vector<uint32_t> cache;  // per device
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        const void *f = (const void *)int4_qkv_tc_kernel<NTOK>;
        cudaFuncSetAttribute(int4_qkv_tc_kernel<NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)I4<NTOK>::kAlloc);
        cache[dev] = (uint32_t)(resident_ctas(f, kThreadsI4, I4<NTOK>::kAlloc, 512) * device_sm_count());
    }
    return cache[dev];
}

cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

template <int NTOK>
cudaError_t launch_i4(const Int4Args &a, const CUtensorMap (&maps)[9], cudaStream_t s) {
    // zero the outputs (the GEMV's CTAs add into them)
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cudaError_t e = launch_int4_zero(a, s);
    if (e != cudaSuccess) return e;
    // one contiguous range of (tile, unit) pairs per CTA: every resident CTA
    // slot, and more CTAs only when a range would exceed kMaxUnits units
    const uint64_t total = (uint64_t)(a.tiles_q + 2 * a.tiles_kv) * (a.k / kUnitK);
    uint64_t ctas = cta_slots_i4<NTOK>();
    const uint64_t need = (total + I4<NTOK>::kMaxUnits - 1) / I4<NTOK>::kMaxUnits;
    if (ctas < need) ctas = need;
    if (ctas > total) ctas = total;
    if (ctas > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kThreadsI4, 1, 1);
    cfg.dynamicSmemBytes = I4<NTOK>::kAlloc;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, int4_qkv_tc_kernel<NTOK>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                              maps[6], maps[7], maps[8], a);
}

}  // namespace

cudaError_t launch_int4_zero(const Int4Args &a, cudaStream_t s) {
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cudaLaunchConfig_t zc = {};
    const size_t elems = (size_t)a.m * (a.nq + 2 * (size_t)a.nkv);
    zc.gridDim = dim3((unsigned)((elems + 255) / 256 < 64 ? (elems + 255) / 256 : 64), 1, 1);
    zc.blockDim = dim3(256, 1, 1);
    zc.stream = s;
    zc.attrs = attr;
    zc.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&zc, int4_zero_kernel, a);
}

bool int4_tc_supported(uint32_t nq, uint32_t nkv, uint32_t group) {
    return group == (uint32_t)kGroupK && nq % 32 == 0 && nkv % 32 == 0;
}

// Two launches (zeroing, then the GEMV) for up to 32 token rows (the API
// passes QDL_INT4_TC_PASS_ROWS at a time).
cudaError_t launch_int4_qkv_tc(const Int4Args &a, cudaStream_t s) {
    CUtensorMap maps[9];
    const uint32_t ns[3] = {a.nq, a.nkv, a.nkv};
    const uint32_t *qw[3] = {a.qw0, a.qw1, a.qw2};
    const float *sc[3] = {a.sc0, a.sc1, a.sc2};
    const float *zr[3] = {a.zr0, a.zr1, a.zr2};
    for (int p = 0; p < 3; ++p) {
        cudaError_t e = make_tmap_4b(&maps[p], CU_TENSOR_MAP_DATA_TYPE_UINT32, qw[p], ns[p] / 8, a.k, kCols / 8, kUnitK,
                                     CU_TENSOR_MAP_SWIZZLE_NONE);
        if (e == cudaSuccess)
            e = make_tmap_4b(&maps[3 + p], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sc[p], ns[p], a.groups, kCols, 1,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
        if (e == cudaSuccess)
            e = make_tmap_4b(&maps[6 + p], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, zr[p], ns[p], a.groups, kCols, 1,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
        if (e != cudaSuccess) return e;
    }
    Int4Args b = a;  // this kernel's tiles are 128 columns wide
    b.tiles_q = (a.nq + kCols - 1) / kCols;
    b.tiles_kv = (a.nkv + kCols - 1) / kCols;
    return a.m <= 16 ? launch_i4<16>(b, maps, s) : launch_i4<32>(b, maps, s);  // the API passes at most QDL_INT4_TC_PASS_ROWS
}

cudaError_t read_and_clear_int4_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_int4_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_int4_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
