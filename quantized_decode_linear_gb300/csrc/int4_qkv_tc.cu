// AWQ INT4 fused Q/K/V projection on the 5th-generation tensor cores
// (fused_int4_qkv.rs: fused_int4_qkv_q, fused_int4_qkv_k, fused_int4_qkv_v,
// unpack_awq_qkv, QKV_AWQ_SHIFTS).  One launch covers all three projections;
// this path serves group size 128 and projection widths that are multiples of
// 32 (the others take the mma.sync kernel in int4_qkv.cu).
//
// Arithmetic (per group g of 128 K values, column c, token m):
//   y[m, c] = sum_g s[g,c] ( sum_{k in g} x~[m,k] (1024 + nib[k,c])
//                            - (1024 + z[g,c]) sum_{k in g} x~[m,k] )
// which equals sum_k x~ (nib - z) s exactly; x~ = x rounded to f16 (the only
// approximation, |x~ - x| <= 2^-11 |x|).  1024 + nib is exact in f16 and is what
// the AWQ bit pattern gives for free: (w >> 4i) & 0x000F000F | 0x64006400 is the
// f16 pair (1024 + nib(col 2i), 1024 + nib(col 2i+1)) of one packed word.
//
// Roles (one CTA = 256 output columns of one projection x a range of groups;
// one pipeline stage = half a group, 64 K rows):
//   warp 0, one lane : TMA producer of the packed words, [64 K rows x 32
//                      words] = 128-byte rows per stage, 128-byte swizzle,
//                      into a ring of stages (evict-first).
//   warp 1           : allocates tensor memory; one lane issues tcgen05.mma
//                      kind::f16, two column halves (M = 128 each) x four
//                      K = 16 steps per stage, N = NTOK tokens; A = weights
//                      MN-major, B = x~ K-major.  The two stages of a group
//                      accumulate into the same TMEM buffer.
//   warps 2..9       : converters.  Unpack each stage's words into the f16 A
//                      operand (a 16-byte load of four words, four 16-byte
//                      stores) and convert x to f16 into the B operand
//                      (128-byte swizzle).
//   warps 10..13     : epilogue.  Per group, read both halves' accumulators
//                      and the all-ones accumulator (= sum x~ per token) with
//                      tcgen05.ld and fold s (acc - (1024 + z) sum x~) into
//                      register totals.
// sum_k x~ comes from one more MMA per K step against a constant all-ones A
// operand, so it is the tensor core's own sum of the same x~.
// Split-K CTAs of one cluster reduce their partials through distributed shared
// memory in rank order.  Every wait is bounded (fault word + drain + return).
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <mutex>
#include <vector>

#include "tma_pipe.cuh"

namespace cg = cooperative_groups;

namespace qdl {

static __device__ uint32_t g_int4_fault;

namespace {

constexpr int kCols = 256;             // output columns per tile (two MMA halves of 128)
constexpr int kGroupK = 128;           // group size
constexpr int kStageK = 64;            // K rows per pipeline stage (half a group)
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreadsI4 = (2 + kConvWarps + kEpiWarps) * 32;
constexpr uint32_t kPacked = kStageK * 128;      // 64 rows x 32 words
constexpr uint32_t kAOp = kCols * kStageK * 2;   // f16 A operand, 32 KB
// A (MN-major, no swizzle): core matrix (8 k rows x 8 columns x 2 B = 128 B)
// (mi, ki) at mi * kAStrideM + ki * kAStrideK
constexpr uint32_t kAStrideM = 128;   // next 8 columns
constexpr uint32_t kAStrideK = 4096;  // next 8 k (32 core matrices of columns)
// all-ones A operand for the per-token sums: 16 x 2 core matrices (M = 128, K = 16)
constexpr uint32_t kOnesStrideK = 2048;
constexpr uint32_t kOnes = 2 * kOnesStrideK;

template <int NTOK>
struct I4 {
    static constexpr uint32_t kXBox = NTOK * 128;                // one x box: NTOK rows x 32 f32 (128-byte swizzle)
    static constexpr uint32_t kRingStage = kPacked + 2 * kXBox;  // packed words + x for 64 K
    static constexpr int kRing = NTOK <= 16 ? 6 : 4;             // ring stages
    static constexpr uint32_t kBOp = NTOK * 128;                 // f16 B operand: one SW128 atom of NTOK rows
    static constexpr uint32_t kOpBuf = kAOp + (kBOp + 1023) / 1024 * 1024;  // one operand buffer (A then B)
    static constexpr int kOps = NTOK <= 16 ? 4 : 3;              // operand buffers: converters run ahead
    static constexpr int kAcc = 4;                               // accumulator buffers (one per group)
    static constexpr uint32_t kRingOff = 0;
    static constexpr uint32_t kOpOff = kRing * kRingStage;
    static constexpr uint32_t kOnesOff = kOpOff + kOps * kOpBuf;  // all-ones A operand, M=128 x K=16
    static constexpr uint32_t kBarOff = kOnesOff + kOnes;
    static constexpr uint32_t kBytes = kBarOff + 512;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static constexpr int kCpt = NTOK;  // token columns per epilogue thread and half
    // per accumulator buffer: column half 0, column half 1, all-ones (sum x~)
    static constexpr uint32_t kTmemCols = 3 * NTOK * kAcc <= 64 ? 64 : (3 * NTOK * kAcc <= 128 ? 128 : (3 * NTOK * kAcc <= 256 ? 256 : 512));
    static_assert(NTOK <= 32, "tokens per pass");
    static_assert(kCols * NTOK * 4 <= kOpOff, "reduction buffer fits the ring");
    static_assert(kOpOff % 1024 == 0 && kOpBuf % 1024 == 0, "alignment");
    static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// MN-major operand without swizzle: the leading byte offset is the stride
// between core matrices along K, the stride byte offset the stride along M
// (measured on sm_103a with an operand whose nibbles encode their own
// coordinates).
__device__ __forceinline__ uint64_t desc_mn_noswz(uint32_t saddr, uint32_t stride_k = kAStrideK) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(stride_k >> 4) << 16;   // leading byte offset: next 8 k
    d |= (uint64_t)(kAStrideM >> 4) << 32;  // stride byte offset: next 8 columns
    d |= (uint64_t)1 << 46;                 // descriptor version
    return d;                               // swizzle none
}

__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t saddr, uint32_t atom_stride) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(atom_stride >> 4) << 16;  // next 64-element K atom
    d |= (uint64_t)(1024 >> 4) << 32;         // next 8 rows
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;                   // 128-byte swizzle
    return d;
}

// kind::f16: D f32, A and B f16, A MN-major (transposed), B K-major.
template <int NTOK>
__device__ __forceinline__ constexpr uint32_t idesc_f16() {
    return (1u << 4) | (1u << 15) | ((uint32_t)(NTOK >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

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

template <int NTOK>
__global__ void __launch_bounds__(kThreadsI4, 1)
    int4_qkv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_x,
                       const Int4Args a) {
    using C = I4<NTOK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);  // [kRing] packed words and x landed
    uint64_t *empty = full + C::kRing;                                  // [kRing] packed slot free
    uint64_t *opfull = empty + C::kRing;                                // [kOps] operands written
    uint64_t *opempty = opfull + C::kOps;                               // [kOps] operands consumed
    uint64_t *accf = opempty + C::kOps;                                 // [kAcc] group accumulated
    uint64_t *acce = accf + C::kAcc;                                    // [kAcc] group drained
    uint64_t *done = acce + C::kAcc;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    float *red = reinterpret_cast<float *>(smem);  // [NTOK][256] at the end

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
    const uint32_t col0 = tile * kCols;
    const uint32_t split = gridDim.y, sidx = blockIdx.y;
    const uint32_t g0 = (a.groups * sidx) / split, g1 = (a.groups * (sidx + 1)) / split;
    const uint32_t ngroups = g1 - g0;
    const uint32_t nstage = 2 * ngroups;  // two stages of 64 K rows per group

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kRing; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConvWarps);
        }
        for (int b = 0; b < C::kOps; ++b) {
            mbar_init(&opfull[b], kConvWarps);
            mbar_init(&opempty[b], 1);
        }
        for (int b = 0; b < C::kAcc; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], kEpiWarps);
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
    // token rows >= m of every B operand stay zero for the whole kernel; the
    // all-ones operand is written once (f16 1.0 = 0x3C00)
    for (uint32_t i = threadIdx.x; i < C::kOps * C::kBOp / 16; i += blockDim.x) {
        const uint32_t buf = i / (C::kBOp / 16), off = (i % (C::kBOp / 16)) * 16;
        *reinterpret_cast<uint4 *>(smem + C::kOpOff + buf * C::kOpBuf + kAOp + off) = make_uint4(0, 0, 0, 0);
    }
    for (uint32_t i = threadIdx.x; i < kOnes / 16; i += blockDim.x)
        *reinterpret_cast<uint4 *>(smem + C::kOnesOff + i * 16) =
            make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fault = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(&g_int4_fault, code);
    };
    auto wait = [&](uint64_t *bar, uint32_t parity, uint32_t code) {
        if (!*abort_flag && !mbar_wait(bar, parity, kWaitLimitNs)) fault(code);
    };

    uint32_t issued = 0;
    float total[2][C::kCpt];  // [column half][token]
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int j = 0; j < C::kCpt; ++j) total[hh][j] = 0.0f;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(tmap);
            prefetch_tmap(&tm_x);
            const uint64_t pol = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            for (uint32_t st = 0; st < nstage; ++st) {
                const uint32_t slot = st % C::kRing, ph = (st / C::kRing) & 1;
                wait(&empty[slot], ph ^ 1, 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], C::kRingStage);
                issued = st + 1;
                uint8_t *rs = smem + C::kRingOff + slot * C::kRingStage;
                const int32_t k0 = (int32_t)(g0 * kGroupK + st * kStageK);
                tma_load_2d(rs, tmap, (int32_t)(col0 / 8), k0, &full[slot], pol);
                tma_load_2d(rs + kPacked, &tm_x, k0, 0, &full[slot], pol_x);            // x[:, k0 .. k0+31]
                tma_load_2d(rs + kPacked + C::kXBox, &tm_x, k0 + 32, 0, &full[slot], pol_x);  // x[:, k0+32 .. k0+63]
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16<NTOK>();
            const uint32_t obase = smem_u32(smem + C::kOpOff);
            const uint32_t ones = smem_u32(smem + C::kOnesOff);
            for (uint32_t st = 0; st < nstage; ++st) {
                const uint32_t o = st % C::kOps, gi = st >> 1, b = gi % C::kAcc, half_k = st & 1;
                if (half_k == 0) wait(&acce[b], ((gi / C::kAcc) & 1) ^ 1, 2);
                wait(&opfull[o], (st / C::kOps) & 1, 4);
                if (*abort_flag) break;
                fence_after();
                const uint32_t abuf = obase + o * C::kOpBuf, bbuf = abuf + kAOp;
                const uint32_t dbase = tmem + b * 3 * NTOK;
#pragma unroll
                for (int i = 0; i < kStageK / 16; ++i) {
                    // A: +16 k = two core matrices along K; B: 32 bytes inside the 64-element atom
                    const uint64_t bd = desc_k_sw128(bbuf + i * 32, NTOK * 128);
                    const uint32_t acc = (half_k | i) != 0 ? 1u : 0u;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)  // column halves
                        mma_f16(dbase + hh * NTOK, desc_mn_noswz(abuf + hh * 16 * kAStrideM + i * 2 * kAStrideK), bd,
                                idesc, acc);
                    mma_f16(dbase + 2 * NTOK, desc_mn_noswz(ones, kOnesStrideK), bd, idesc, acc);  // sum x~
                }
                commit(&opempty[o]);
                if (half_k == 1) commit(&accf[b]);
            }
            commit(done);
        }
    } else if (warp < 2 + kConvWarps) {
        // ------------------------------------------------------------ converters
        const int t = threadIdx.x - 64;                   // 0 .. 255
        const uint32_t kr = t & 7, wq = (t >> 3) & 7, kq = t >> 6;  // K row in a core matrix, word quad, K quarter
        for (uint32_t st = 0; st < nstage; ++st) {
            const uint32_t slot = st % C::kRing, ph = (st / C::kRing) & 1;
            const uint32_t o = st % C::kOps;
            wait(&opempty[o], ((st / C::kOps) & 1) ^ 1, 16);
            wait(&full[slot], ph, 16);
            // A: words (k, 4wq .. 4wq+3) for k = 8 (kq + 4j) + kr: one 16-byte load,
            // then row k & 7 of core matrices (4wq + i, k / 8).  Plain shared-memory
            // accesses (ordered by the barrier waits' memory clobbers).
            const uint8_t *ring = smem + C::kRingOff + slot * C::kRingStage;
            uint8_t *abuf = smem + C::kOpOff + o * C::kOpBuf;
            uint4 wv[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t k = 8 * (kq + 4 * j) + kr;
                // 128-byte swizzle of the TMA tile: 16-byte chunk index ^= row & 7
                wv[j] = *reinterpret_cast<const uint4 *>(ring + k * 128 + ((wq ^ (k & 7)) << 4));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t k = 8 * (kq + 4 * j) + kr;
                const uint32_t w4[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t w = w4[i];  // words beyond the projection width read as zero (TMA fill)
                    uint4 h;
                    h.x = (w & 0x000F000Fu) | 0x64006400u;
                    h.y = ((w >> 4) & 0x000F000Fu) | 0x64006400u;
                    h.z = ((w >> 8) & 0x000F000Fu) | 0x64006400u;
                    h.w = ((w >> 12) & 0x000F000Fu) | 0x64006400u;
                    *reinterpret_cast<uint4 *>(abuf + (4 * wq + i) * kAStrideM + (k >> 3) * kAStrideK + kr * 16) = h;
                }
            }
            // B: x~ (f16) in the K-major 128-byte-swizzle layout.  x of this stage
            // sits in the ring stage as two [NTOK x 32 f32] boxes (128-byte
            // swizzle); only valid token rows are written.
            uint8_t *bbuf = abuf + kAOp;
#pragma unroll
            for (int i = 0; i < NTOK / 8; ++i) {
                const uint32_t tok = (t & 7) + 8 * i;
                const uint32_t kc = t >> 3;  // 8-value chunk 0..7 of the stage; threads with kc >= 8 idle
                if (kc < 8 && tok < a.m) {
                    const uint8_t *xb = ring + kPacked + (kc >> 2) * C::kXBox + tok * 128;
                    const uint32_t c0 = (2 * (kc & 3)) ^ (tok & 7), c1 = (2 * (kc & 3) + 1) ^ (tok & 7);
                    const float4 u = *reinterpret_cast<const float4 *>(xb + (c0 << 4));
                    const float4 v = *reinterpret_cast<const float4 *>(xb + (c1 << 4));
                    *reinterpret_cast<uint4 *>(bbuf + tok * 128 + ((kc ^ (tok & 7)) << 4)) =
                        make_uint4(h2_bits(u.x, u.y), h2_bits(u.z, u.w), h2_bits(v.x, v.y), h2_bits(v.z, v.w));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[slot]);  // ring stage (words and x) consumed
                mbar_arrive(&opfull[o]);    // operands written
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const uint32_t lrow = 32 * quad + lane;  // column within a half
        const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
        for (uint32_t gi = 0; gi < ngroups; ++gi) {
            const uint32_t b = gi % C::kAcc, g = g0 + gi;
            float s_c[2], zc[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t col = col0 + hh * 128 + lrow;
                const bool ok = col < n;
                s_c[hh] = ok ? __ldg(sc + (size_t)g * n + col) : 0.0f;
                zc[hh] = 1024.0f + (ok ? __ldg(zr + (size_t)g * n + col) : 0.0f);
            }
            wait(&accf[b], (gi / C::kAcc) & 1, 32);
            fence_after();
#pragma unroll
            for (int c = 0; c < C::kCpt / 16; ++c) {
                float sx[16], v0[16], v1[16];
                ld16(taddr + b * 3 * NTOK + 2 * NTOK + 16 * c, sx);  // sum x~ per token (any row)
                ld16(taddr + b * 3 * NTOK + 16 * c, v0);
                ld16(taddr + b * 3 * NTOK + NTOK + 16 * c, v1);
                wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    total[0][16 * c + i] = fmaf(s_c[0], fmaf(-zc[0], sx[i], v0[i]), total[0][16 * c + i]);
                    total[1][16 * c + i] = fmaf(s_c[1], fmaf(-zc[1], sx[i], v1[i]), total[1][16 * c + i]);
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
        }
    }

    // ---------------------------------------------------------------- drain after a timeout
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t first = issued > (uint32_t)C::kRing ? issued - C::kRing : 0;
            for (uint32_t st = first; st < issued; ++st)
                mbar_wait(&full[st % C::kRing], (st / C::kRing) & 1, kWaitLimitNs);
        }
        if (warp == 1 && lane == 0) mbar_wait(done, 0, kWaitLimitNs);
        __syncthreads();
    }

    auto store = [&](uint32_t tok, uint32_t lc, float v) {
        if (tok < a.m && col0 + lc < n) out[(size_t)tok * n + col0 + lc] = v;
    };
    if (warp >= 2 + kConvWarps) {
        const uint32_t lrow = 32 * (warp & 3) + lane;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int j = 0; j < C::kCpt; ++j) {
                if (split == 1)
                    store(j, hh * 128 + lrow, total[hh][j]);
                else
                    red[j * kCols + hh * 128 + lrow] = total[hh][j];
            }
    }
    if (split > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const uint32_t c_lo = (kCols * sidx) / split, c_hi = (kCols * (sidx + 1)) / split;
        const uint32_t span = c_hi - c_lo;
        const uint32_t m_used = a.m < (uint32_t)NTOK ? a.m : (uint32_t)NTOK;
        const float *peer[8];
#pragma unroll
        for (int rk = 0; rk < 8; ++rk) peer[rk] = cluster.map_shared_rank(red, rk < (int)split ? rk : 0);
        for (uint32_t idx = threadIdx.x; idx < span * m_used; idx += blockDim.x) {
            const uint32_t tok = idx / span, lc = c_lo + idx % span;
            float v[8];
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) v[rk] = rk < (int)split ? peer[rk][tok * kCols + lc] : 0.0f;
            float s = 0.0f;
#pragma unroll
            for (int rk = 0; rk < 8; ++rk) s += v[rk];
            store(tok, lc, s);
        }
        cluster.sync();
    }

    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

template <int NTOK>
const uint32_t *cluster_fit() {
    static std::mutex mu;
    static std::vector<std::vector<uint32_t>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    if (cache[dev].empty()) {
        const void *f = (const void *)int4_qkv_tc_kernel<NTOK>;
        cudaFuncSetAttribute(int4_qkv_tc_kernel<NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)I4<NTOK>::kAlloc);
        const int per_sm = resident_ctas(f, kThreadsI4, I4<NTOK>::kAlloc, I4<NTOK>::kTmemCols);
        cache[dev].assign(8, 0);
        resident_cta_slots(f, kThreadsI4, I4<NTOK>::kAlloc, per_sm, cache[dev].data());
    }
    return cache[dev].data();
}

template <int NTOK>
cudaError_t launch_i4(const Int4Args &a, const CUtensorMap (&maps)[4], cudaStream_t s) {
    const uint32_t tiles = a.tiles_q + 2 * a.tiles_kv;
    const uint32_t split = choose_split_k(tiles, a.groups, cluster_fit<NTOK>(), 0.0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, split, 1);
    cfg.blockDim = dim3(kThreadsI4, 1, 1);
    cfg.dynamicSmemBytes = I4<NTOK>::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, int4_qkv_tc_kernel<NTOK>, maps[0], maps[1], maps[2], maps[3], a);
}

}  // namespace

cudaError_t make_tmap_words(CUtensorMap *map, const void *base, uint64_t words, uint64_t rows, uint32_t box_rows) {
    // packed words [rows, words] u32, box 32 words x box_rows rows, 128-byte swizzle
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
    if (fn == nullptr) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {words, rows};
    cuuint64_t gstride[1] = {words * 4};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_f32(CUtensorMap *map, const float *x, uint64_t k, uint64_t rows, uint32_t box_rows) {
    // x [rows, k] f32, box 32 values x box_rows rows, 128-byte swizzle; rows
    // past the end read as zero
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
    if (fn == nullptr) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {k, rows};
    cuuint64_t gstride[1] = {k * 4};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(x), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}



bool int4_tc_supported(uint32_t nq, uint32_t nkv, uint32_t group) {
    return group == (uint32_t)kGroupK && nq % 32 == 0 && nkv % 32 == 0;
}

// One launch for up to 32 token rows.
cudaError_t launch_int4_qkv_tc(const Int4Args &a, cudaStream_t s) {
    CUtensorMap maps[4];
    const uint32_t ns[3] = {a.nq, a.nkv, a.nkv};
    const uint32_t *qw[3] = {a.qw0, a.qw1, a.qw2};
    for (int p = 0; p < 3; ++p) {
        cudaError_t e = make_tmap_words(&maps[p], qw[p], ns[p] / 8, a.k, kStageK);
        if (e != cudaSuccess) return e;
    }
    const uint32_t ntok = a.m <= 16 ? 16 : 32;
    cudaError_t e = make_tmap_f32(&maps[3], a.x, a.k, a.m, ntok);
    if (e != cudaSuccess) return e;
    Int4Args b = a;  // this kernel's tiles are 256 columns wide
    b.tiles_q = (a.nq + kCols - 1) / kCols;
    b.tiles_kv = (a.nkv + kCols - 1) / kCols;
    return ntok == 16 ? launch_i4<16>(b, maps, s) : launch_i4<32>(b, maps, s);
}

cudaError_t read_and_clear_int4_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_int4_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_int4_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
