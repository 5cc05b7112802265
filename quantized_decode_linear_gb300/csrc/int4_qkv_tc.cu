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
// Roles (one CTA = 128 output columns of one projection x a range of groups):
//   warp 0, one lane : TMA producer of the packed words, [128 K rows x 16
//                      words] per group, 64-byte swizzle, into a ring of
//                      stages (evict-first).
//   warp 1           : allocates tensor memory; one lane issues tcgen05.mma
//                      kind::f16 (M = 128 columns, N = NTOK tokens, K = 16 per
//                      instruction, eight per group), A = weights MN-major,
//                      B = x~ K-major.
//   warps 2..9       : converters.  Unpack each group's words into the f16 A
//                      operand (one 16-byte store per word), convert the group's
//                      x to f16 into the B operand (128-byte swizzle) and sum
//                      x~ per token (fixed order).
//   warps 10..13     : epilogue.  Per group, read the accumulator (tcgen05.ld)
//                      and fold s (acc - (1024 + z) sum x~) into register
//                      totals.
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

constexpr int kCols = 128;             // output columns per tile (MMA M)
constexpr int kGroupK = 128;           // K per stage = group size
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreadsI4 = (2 + kConvWarps + kEpiWarps) * 32;
constexpr uint32_t kPacked = kGroupK * 64;  // 128 rows x 16 words
constexpr uint32_t kAOp = kCols * kGroupK * 2;  // f16 A operand, 32 KB
// A (MN-major, no swizzle): core matrix (8 k rows x 8 columns x 2 B = 128 B)
// (mi, ki) at mi * kAStrideM + ki * kAStrideK
constexpr uint32_t kAStrideM = 128;   // next 8 columns
constexpr uint32_t kAStrideK = 2048;  // next 8 k

template <int NTOK>
struct I4 {
    static constexpr int kRing = 8;                              // packed stages
    static constexpr uint32_t kBOp = NTOK * 256;                 // f16 B operand: 2 SW128 atoms of NTOK rows
    static constexpr uint32_t kOpBuf = kAOp + kBOp;              // one operand buffer (A then B)
    static constexpr int kAcc = NTOK <= 64 ? 4 : 2;
    static constexpr uint32_t kRingOff = 0;
    static constexpr uint32_t kOpOff = kRing * kPacked;          // 64 KB
    static constexpr uint32_t kBarOff = kOpOff + 2 * kOpBuf;
    static constexpr uint32_t kSumOff = kBarOff + 512;           // [kAcc][NTOK] sum x~
    static constexpr uint32_t kPartOff = kSumOff + kAcc * NTOK * 4;  // [NTOK][16] partial sums
    static constexpr uint32_t kBytes = kPartOff + NTOK * 16 * 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static constexpr int kCpt = NTOK;  // columns per epilogue thread (NTOK <= 64)
    static constexpr uint32_t kTmemCols = NTOK * kAcc <= 32 ? 32 : (NTOK * kAcc <= 64 ? 64 : (NTOK * kAcc <= 128 ? 128 : 256));
    static_assert(NTOK <= 32, "tokens per pass");
    static_assert(kCols * NTOK * 4 <= kOpOff, "reduction buffer fits the ring");
    static_assert(kOpOff % 1024 == 0 && kOpBuf % 1024 == 0, "alignment");
};

// MN-major operand without swizzle: the leading byte offset is the stride
// between core matrices along K, the stride byte offset the stride along M
// (measured on sm_103a with an operand whose nibbles encode their own
// coordinates).
__device__ __forceinline__ uint64_t desc_mn_noswz(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(kAStrideK >> 4) << 16;  // leading byte offset: next 8 k
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
    return (1u << 4) | (1u << 15) | ((uint32_t)(NTOK >> 3) << 17) | ((uint32_t)(kCols >> 4) << 24);
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

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void conv_barrier() {  // the converter warps only
    asm volatile("bar.sync 1, %0;" ::"n"(kConvWarps * 32) : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int NTOK>
__global__ void __launch_bounds__(kThreadsI4, 1)
    int4_qkv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const Int4Args a) {
    using C = I4<NTOK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);  // [kRing] packed words landed
    uint64_t *empty = full + C::kRing;                                  // [kRing] packed slot free
    uint64_t *opfull = empty + C::kRing;                                // [2] operands written
    uint64_t *opempty = opfull + 2;                                     // [2] operands consumed
    uint64_t *accf = opempty + 2;                                       // [kAcc]
    uint64_t *acce = accf + C::kAcc;                                    // [kAcc]
    uint64_t *sums = acce + C::kAcc;                                    // [kAcc] sum x~ written
    uint64_t *done = sums + C::kAcc;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    float *sbuf = reinterpret_cast<float *>(smem + C::kSumOff);
    float *part = reinterpret_cast<float *>(smem + C::kPartOff);
    float *red = reinterpret_cast<float *>(smem);  // [NTOK][128] at the end

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
    const uint32_t niter = g1 - g0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kRing; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConvWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&opfull[b], kConvWarps);
            mbar_init(&opempty[b], 1);
        }
        for (int b = 0; b < C::kAcc; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], kEpiWarps);
            mbar_init(&sums[b], 1);
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
    // token rows >= m of both B operands stay zero for the whole kernel
    for (uint32_t i = threadIdx.x; i < 2 * C::kBOp / 16; i += blockDim.x) {
        const uint32_t buf = i / (C::kBOp / 16), off = (i % (C::kBOp / 16)) * 16;
        sts128(smem_u32(smem + C::kOpOff + buf * C::kOpBuf + kAOp + off), 0, 0, 0, 0);
    }
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
    float total[C::kCpt];
#pragma unroll
    for (int j = 0; j < C::kCpt; ++j) total[j] = 0.0f;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(tmap);
            const uint64_t pol = policy_evict_first();
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t slot = it % C::kRing, ph = (it / C::kRing) & 1;
                wait(&empty[slot], ph ^ 1, 1);
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[slot], kPacked);
                issued = it + 1;
                tma_load_2d(smem + C::kRingOff + slot * kPacked, tmap, (int32_t)(col0 / 8),
                            (int32_t)((g0 + it) * kGroupK), &full[slot], pol);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16<NTOK>();
            const uint32_t obase = smem_u32(smem + C::kOpOff);
            for (uint32_t it = 0; it < niter; ++it) {
                const uint32_t o = it & 1, b = it % C::kAcc;
                wait(&acce[b], ((it / C::kAcc) & 1) ^ 1, 2);
                wait(&opfull[o], (it >> 1) & 1, 4);
                if (*abort_flag) break;
                fence_after();
                const uint32_t abuf = obase + o * C::kOpBuf, bbuf = abuf + kAOp;
#pragma unroll
                for (int i = 0; i < kGroupK / 16; ++i) {
                    // A: +16 k = two core matrices along K; B: 32 bytes inside a
                    // 64-element atom, next atom every four instructions
                    const uint64_t ad = desc_mn_noswz(abuf + i * 2 * kAStrideK);
                    const uint64_t bd = desc_k_sw128(bbuf + (i >> 2) * (NTOK * 128) + (i & 3) * 32, NTOK * 128);
                    mma_f16(tmem + b * NTOK, ad, bd, idesc, i > 0 ? 1u : 0u);
                }
                commit(&opempty[o]);
                commit(&accf[b]);
            }
            commit(done);
        }
    } else if (warp < 2 + kConvWarps) {
        // ------------------------------------------------------------ converters
        const int t = threadIdx.x - 64;  // 0 .. 255
        const uint32_t kl = t & 7, wc = (t >> 3) & 15, kh = t >> 7;
        const uint32_t rbase = smem_u32(smem + C::kRingOff);
        const uint32_t obase = smem_u32(smem + C::kOpOff);
        const bool word_ok = col0 / 8 + wc < n / 8;
        for (uint32_t it = 0; it < niter; ++it) {
            const uint32_t slot = it % C::kRing, ph = (it / C::kRing) & 1;
            const uint32_t o = it & 1, b = it % C::kAcc;
            const uint32_t g = g0 + it;
            // x for this group: token tok = (t & 7) + 8i, 8 K values at chunk t >> 3 (0..15 -> 16 x 8 = 128)
            float4 xv[NTOK / 8][2];
#pragma unroll
            for (int i = 0; i < NTOK / 8; ++i) {
                const uint32_t tok = (t & 7) + 8 * i;
                const uint32_t kc = t >> 3;
                if (tok < a.m && kc < 16) {
                    const float4 *p = reinterpret_cast<const float4 *>(a.x + (size_t)tok * a.k + g * kGroupK + kc * 8);
                    xv[i][0] = __ldg(p);
                    xv[i][1] = __ldg(p + 1);
                } else {
                    xv[i][0] = xv[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            wait(&opempty[o], ((it >> 1) & 1) ^ 1, 16);
            wait(&acce[b], ((it / C::kAcc) & 1) ^ 1, 16);
            wait(&full[slot], ph, 16);
            // A: words (k, wc) for k = 8 (2j + kh) + kl -> 16-byte row kl of core matrix (wc, k / 8)
            const uint32_t ring = rbase + slot * kPacked;
            const uint32_t abuf = obase + o * C::kOpBuf;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t k = 8 * (2 * j + kh) + kl;
                // 64-byte swizzle of the TMA tile: 16-byte chunk index ^= (row >> 1) & 3
                const uint32_t w = word_ok ? lds32(ring + k * 64 + ((((wc >> 2) ^ ((k >> 1) & 3))) << 4) + (wc & 3) * 4)
                                           : 0u;
                uint32_t h[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) h[i] = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
                sts128(abuf + wc * kAStrideM + (k >> 3) * kAStrideK + kl * 16, h[0], h[1], h[2], h[3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);  // packed words consumed
            // B: x~ (f16) in the K-major 128-byte-swizzle layout, plus partial sums
            const uint32_t bbuf = abuf + kAOp;
#pragma unroll
            for (int i = 0; i < NTOK / 8; ++i) {
                const uint32_t tok = (t & 7) + 8 * i;
                const uint32_t kc = t >> 3;  // 0..31; chunks >= 16 idle
                if (kc < 16) {
                    const float4 u = xv[i][0], v = xv[i][1];
                    const uint32_t p0 = h2_bits(u.x, u.y), p1 = h2_bits(u.z, u.w), p2 = h2_bits(v.x, v.y),
                                   p3 = h2_bits(v.z, v.w);
                    if (tok < a.m) {
                        const uint32_t atom = kc >> 3, chunk = kc & 7;
                        sts128(bbuf + atom * (NTOK * 128) + tok * 128 + ((chunk ^ (tok & 7)) << 4), p0, p1, p2, p3);
                    }
                    // partial sum of the rounded values, in a fixed order
                    const __half2 *hp0 = reinterpret_cast<const __half2 *>(&p0);
                    const __half2 *hp1 = reinterpret_cast<const __half2 *>(&p1);
                    const __half2 *hp2 = reinterpret_cast<const __half2 *>(&p2);
                    const __half2 *hp3 = reinterpret_cast<const __half2 *>(&p3);
                    float ps = 0.0f;
                    ps += __low2float(*hp0); ps += __high2float(*hp0);
                    ps += __low2float(*hp1); ps += __high2float(*hp1);
                    ps += __low2float(*hp2); ps += __high2float(*hp2);
                    ps += __low2float(*hp3); ps += __high2float(*hp3);
                    part[tok * 16 + kc] = ps;
                }
            }
            fence_proxy_async_smem();
            conv_barrier();
            if (t < NTOK) {  // sum x~ of token t over the group's 16 chunks, in order
                float s = 0.0f;
#pragma unroll
                for (int c = 0; c < 16; ++c) s += part[t * 16 + c];
                sbuf[b * NTOK + t] = s;
            }
            conv_barrier();
            __syncwarp();
            if (lane == 0) mbar_arrive(&opfull[o]);
            if (t == 0) mbar_arrive(&sums[b]);
            (void)g;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const uint32_t lrow = 32 * quad + lane;  // column within the tile
        const uint32_t col = col0 + lrow;
        const bool col_ok = col < n;
        const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
        for (uint32_t it = 0; it < niter; ++it) {
            const uint32_t b = it % C::kAcc, g = g0 + it;
            const float s_c = col_ok ? __ldg(sc + (size_t)g * n + col) : 0.0f;
            const float z_c = col_ok ? __ldg(zr + (size_t)g * n + col) : 0.0f;
            const float zc = 1024.0f + z_c;
            wait(&sums[b], (it / C::kAcc) & 1, 32);
            wait(&accf[b], (it / C::kAcc) & 1, 32);
            fence_after();
#pragma unroll
            for (int c = 0; c < C::kCpt / 16; ++c) {
                float v[16];
                ld16(taddr + b * NTOK + 16 * c, v);
                wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float sx = sbuf[b * NTOK + 16 * c + i];
                    total[16 * c + i] = fmaf(s_c, fmaf(-zc, sx, v[i]), total[16 * c + i]);
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
            for (uint32_t it = first; it < issued; ++it)
                mbar_wait(&full[it % C::kRing], (it / C::kRing) & 1, kWaitLimitNs);
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
        for (int j = 0; j < C::kCpt; ++j) {
            if (split == 1)
                store(j, lrow, total[j]);
            else
                red[j * kCols + lrow] = total[j];
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

cudaError_t make_tmap_words(CUtensorMap *map, const void *base, uint64_t words, uint64_t rows) {
    // packed words [rows, words] u32, box 16 words x 128 rows, 64-byte swizzle
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
    cuuint32_t box[2] = {16, (cuuint32_t)kGroupK};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NTOK>
uint32_t slots_i4() {
    static std::mutex mu;
    static std::vector<uint32_t> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        cudaFuncSetAttribute(int4_qkv_tc_kernel<NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)I4<NTOK>::kAlloc);
        cache[dev] = (uint32_t)(device_sm_count() * resident_ctas((const void *)int4_qkv_tc_kernel<NTOK>, kThreadsI4,
                                                                  I4<NTOK>::kAlloc, I4<NTOK>::kTmemCols));
    }
    return cache[dev];
}

template <int NTOK>
cudaError_t launch_i4(const Int4Args &a, const CUtensorMap (&maps)[3], cudaStream_t s) {
    const uint32_t tiles = a.tiles_q + 2 * a.tiles_kv;
    const uint32_t split = choose_split_k(tiles, a.groups, slots_i4<NTOK>());
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
    return cudaLaunchKernelEx(&cfg, int4_qkv_tc_kernel<NTOK>, maps[0], maps[1], maps[2], a);
}

}  // namespace

bool int4_tc_supported(uint32_t nq, uint32_t nkv, uint32_t group) {
    return group == (uint32_t)kGroupK && nq % 32 == 0 && nkv % 32 == 0;
}

// One launch for up to 32 token rows.
cudaError_t launch_int4_qkv_tc(const Int4Args &a, cudaStream_t s) {
    CUtensorMap maps[3];
    const uint32_t ns[3] = {a.nq, a.nkv, a.nkv};
    const uint32_t *qw[3] = {a.qw0, a.qw1, a.qw2};
    for (int p = 0; p < 3; ++p) {
        cudaError_t e = make_tmap_words(&maps[p], qw[p], ns[p] / 8, a.k);
        if (e != cudaSuccess) return e;
    }
    return a.m <= 16 ? launch_i4<16>(a, maps, s) : launch_i4<32>(a, maps, s);
}

cudaError_t read_and_clear_int4_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_int4_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_int4_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
