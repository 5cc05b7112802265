// AWQ INT4 fused Q/K/V projection for a few token rows on the CUDA cores
// (fused_int4_qkv.rs: fused_int4_qkv_q, fused_int4_qkv_k, fused_int4_qkv_v,
// unpack_awq_qkv, QKV_AWQ_SHIFTS).  One launch covers all three projections,
// 1 to 8 token rows, any group that is a multiple of 16; a zeroing launch
// goes first, since CTAs add their totals into the outputs.
//
// With one to a few tokens every weight is used once or a few times, so the
// work is a stream of 4-bit codes that has to reach every SM at once and be
// turned into products with as few instructions per code as possible.
//
// Arithmetic (per group g, column c, token t):
//   y[t, c] = sum_g s[g,c] ( sum_{k in g} x[t,k] nib[k,c] - z[g,c] sum_{k in g} x[t,k] )
// which is sum_k x (nib - z) s regrouped; x stays f32, nib is exact, the inner
// sums accumulate in f32.  The regrouping holds for any run of K rows inside
// one group, so each 32-row stage (or 16-row half, where a group ends there)
// is folded on its own.  A nibble at bit 4e of a word (e <= 4) becomes the
// float nib * 16^e exactly: OR its masked bits into the pattern of 2^23 and
// subtract 2^23 (one lop3, and half of one paired f32 add).  The 16^-e factor
// is applied to s at the fold, where it is exact (a power of two).  The AWQ
// word holds columns {0, 2, 4, 6, 1, 3, 5, 7} at nibbles 0..7 (shifts
// {0,16,4,20,8,24,12,28} of columns 0..7); nibbles 5..7 are read from the
// word shifted right by 12.  Products and sums run on packed f32 pairs
// (fma.rn.f32x2 / add.rn.f32x2): two nibbles of one word per instruction,
// each rounded exactly as the scalar f32 operation would be.
//
// Work split (stream-K): a tile is 256 output columns (32 packed words) of one
// projection; a stage is 32 K rows of one tile (4 KB of codes).  The stages
// of all tiles, tile-major, are cut into one contiguous range per CTA, one CTA
// per SM (more CTAs only where a range would not fit the CTA's shared memory),
// so every SM streams the same number of code bytes.  The producer requests
// every stage of the range at once: the codes before the kernel waits for the
// previous one, x after it.  Inside a CTA the range's 16-row halves are split
// evenly into one contiguous slice per consumer warp, so all warps finish
// together; a warp waits only for the stages its slice touches.
//
// Roles:
//   warp 0           : TMA producer (one lane per stage for 1-2 tokens,
//                      lane 0 for all stages otherwise): the stage's
//                      [32 rows x 32 words] codes, and its [tokens x 32] box
//                      of x after the dependency wait.
//   warps 1..C       : consumers; lane l owns word column l (8 output
//                      columns).  Per 16-row half: the 16 code words are
//                      loaded first, then converted and multiplied.  Sums
//                      are folded with the group's scale and zero when the
//                      group (or tile) changes; the next group's scales and
//                      zeros are loaded one group ahead.  Folded sums stay in
//                      registers while the warp stays on one tile and go to a
//                      shared per-tile area (shared f32 adds; the lane's 8
//                      columns padded to 9, so a warp's adds hit distinct
//                      banks) when it moves to another tile and at the end.
// At the end the CTA adds each tile's totals into the outputs with one
// vector f32 atomic add per 4 columns.  Unit positions are walked
// incrementally (no integer division per stage).  Every wait is bounded
// (fault word, drain, return).
#include <mutex>
#include <vector>

#include "tma_pipe.cuh"

namespace qdl {

static __device__ uint32_t g_int4cc_fault;

namespace {

constexpr int kColsS = 256;                    // output columns per tile (32 words)
constexpr uint32_t kRowsS = 32;                // K rows per stage
constexpr uint32_t kCodeBytes = kRowsS * 128;  // 4 KB of packed codes per stage
constexpr uint32_t kStageS = 5120;             // codes + x box (up to 8 tokens x 32 f32)
#ifndef QDL_INT4_SK_STAGES
#define QDL_INT4_SK_STAGES 36  // stages resident per CTA (a CTA's whole range)
#endif
#ifndef QDL_INT4_SK_EARLY
// 1: release dependent kernels at the start (before the dependency wait the
// kernel only streams read-only codes), so that the next call's zeroing
// kernel is resident before this one ends.  Measured on the K=4096 QKV
// projection: 9.3 -> 8.3 us at M=1, 13.9 -> 12.3 us at M=4.
#define QDL_INT4_SK_EARLY 1
#endif
#ifndef QDL_INT4_SK_C1
#define QDL_INT4_SK_C1 20  // consumer warps for 1 token (16: 8.3 us, 20: 8.0 us on the QKV workload)
#endif
constexpr int kMaxStages = QDL_INT4_SK_STAGES;
constexpr uint32_t kBarOffS = kMaxStages * kStageS;
constexpr int kMaxSeg = 4;     // tiles one CTA's range may touch
constexpr int kRedPitch = 288; // per (tile, token): 32 lanes x 9 (8 columns + 1 pad)
static_assert((kMaxStages + 2) * 8 <= 1024, "barrier area");

template <int MT>
struct Sk {
    // warps are spread over the SM's four register files: 21 warps leave 80
    // registers a thread (1 token), 16 leave 128 (2 tokens), 12 leave 168
    // (4 tokens), 8 leave 255 (8 tokens)
    static constexpr int kConsumers = MT == 1 ? QDL_INT4_SK_C1 : MT == 2 ? 15 : MT == 4 ? 11 : 7;
    static constexpr int kThreads = (1 + kConsumers) * 32;
    static constexpr uint32_t kRedOff = kBarOffS + 1024;
    static constexpr uint32_t kRedFloats = kMaxSeg * MT * kRedPitch;
    static constexpr uint32_t kAlloc = kRedOff + kRedFloats * 4 + 1024;  // + base alignment slack
    static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// column (within the word) held by physical nibble p, and the exponent e of
// the value nib * 16^e that nibble p is read as
__device__ __forceinline__ constexpr int nib_col(int p) { return p < 4 ? 2 * p : 2 * (p - 4) + 1; }
__device__ __forceinline__ constexpr int nib_exp(int p) { return p <= 4 ? p : p - 3; }

// 2^23 + nib * 16^e: the masked bits of v ORed into the pattern of 2^23
__device__ __forceinline__ float magic_nib(uint32_t v, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(0x4B000000u));  // (v & m) | c
    return __uint_as_float(r);
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Position of a unit: global tile index (projections q, k, v in order) and
// stage within the tile, walked forward without division.
struct Walk {
    uint32_t tile, st;
    __device__ __forceinline__ void advance(uint32_t by, uint32_t stages) {
        st += by;
        while (st >= stages) {
            st -= stages;
            ++tile;
        }
    }
};

// projection and tile within it of global tile t
__device__ __forceinline__ void tile_proj(const Int4Args &a, uint32_t t, uint32_t &proj, uint32_t &tile) {
    if (t < a.tiles_q) {
        proj = 0; tile = t;
    } else if (t < a.tiles_q + a.tiles_kv) {
        proj = 1; tile = t - a.tiles_q;
    } else {
        proj = 2; tile = t - a.tiles_q - a.tiles_kv;
    }
}

template <int MT>
__global__ void __launch_bounds__(Sk<MT>::kThreads, 1)
    int4_qkv_sk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_x,
                       const Int4Args a, const uint32_t stages, const uint32_t base, const uint32_t rem,
                       const uint32_t vec4) {
    using C = Sk<MT>;
    constexpr int kConsumers = C::kConsumers;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // offset into the shared array itself (keeps the shared address space)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kBarOffS);  // [kMaxStages] codes and x landed
    volatile uint32_t *abort_flag = reinterpret_cast<uint32_t *>(full + kMaxStages);
    float *red = reinterpret_cast<float *>(smem + C::kRedOff);       // [kMaxSeg][MT][kRedPitch]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's range of units: `base` each, one more for the first `rem`
    const uint32_t cta = blockIdx.x;
    const uint32_t u_lo = cta * base + (cta < rem ? cta : rem);
    const uint32_t nloc = base + (cta < rem ? 1u : 0u);
    const uint32_t t_first = u_lo / stages;
    const uint32_t st_first = u_lo - t_first * stages;
    const uint32_t nseg = nloc == 0 ? 0 : (st_first + nloc - 1) / stages + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    for (uint32_t i = threadIdx.x; i < C::kRedFloats; i += blockDim.x) red[i] = 0.0f;
    __syncthreads();
    if (QDL_INT4_SK_EARLY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    auto fault = [&](uint32_t code) {
        *abort_flag = 1;
        atomicOr(&g_int4cc_fault, code);
    };

    uint32_t issued = 0;
    if (nseg > (uint32_t)kMaxSeg || nloc > (uint32_t)kMaxStages) {
        if (threadIdx.x == 0) fault(4);  // the launcher sizes ranges so this cannot happen
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        // codes before waiting for the previous kernel (weights are not
        // written by it), x after.  For 1-2 tokens lane l requests stages
        // l, l + 32, ... (one issuing thread took about 1 us for its first
        // copy and 100-150 ns for each further one): 8.1 -> 6.6 us at M = 1,
        // 8.8 -> 7.5 us at M = 2 on the QKV workload.  For more tokens, whose
        // compute is longer, lane 0 requests them in order (11.6 us at M = 4,
        // 12.0 with every lane issuing).
        const uint64_t pol = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        constexpr uint32_t kTx = kCodeBytes + MT * 128;
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_x);
        }
        if constexpr (MT <= 2) {
            Walk w0 = {t_first + (st_first + lane) / stages, (st_first + lane) % stages};
            Walk wk = w0;
            for (uint32_t j = lane; j < nloc; j += 32, wk.advance(32, stages)) {
                uint32_t proj, tile;
                tile_proj(a, wk.tile, proj, tile);
                const CUtensorMap *map = proj == 0 ? &tm_q : proj == 1 ? &tm_k : &tm_v;
                mbar_arrive_expect_tx(&full[j], kTx);
                tma_load_2d(smem + j * kStageS, map, (int32_t)(tile * 32), (int32_t)(wk.st * kRowsS), &full[j], pol);
            }
            issued = nloc;  // every stage was requested (read by lane 0 when draining)
            asm volatile("griddepcontrol.wait;" ::: "memory");  // x and the zeroed outputs come from earlier kernels
            Walk wx = w0;
            for (uint32_t j = lane; j < nloc; j += 32, wx.advance(32, stages))
                tma_load_2d(smem + j * kStageS + kCodeBytes, &tm_x, (int32_t)(wx.st * kRowsS), 0, &full[j], pol_x);
        } else if (lane == 0) {
            const CUtensorMap *maps[3] = {&tm_q, &tm_k, &tm_v};
            Walk wk = {t_first, st_first};
            for (uint32_t j = 0; j < nloc; ++j, wk.advance(1, stages)) {
                uint32_t proj, tile;
                tile_proj(a, wk.tile, proj, tile);
                mbar_arrive_expect_tx(&full[j], kTx);
                issued = j + 1;
                tma_load_2d(smem + j * kStageS, maps[proj], (int32_t)(tile * 32), (int32_t)(wk.st * kRowsS), &full[j],
                            pol);
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");  // x and the zeroed outputs come from earlier kernels
            Walk wx = {t_first, st_first};
            for (uint32_t j = 0; j < nloc; ++j, wx.advance(1, stages))
                tma_load_2d(smem + j * kStageS + kCodeBytes, &tm_x, (int32_t)(wx.st * kRowsS), 0, &full[j], pol_x);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const float2 kMagic = make_float2(-8388608.0f, -8388608.0f);
        const uint32_t cw = (uint32_t)(warp - 1);
        const uint32_t halves = 2 * nloc;
        const uint32_t h_lo = cw * halves / kConsumers, h_hi = (cw + 1) * halves / kConsumers;
        const uint32_t tiles_total = a.tiles_q + 2 * a.tiles_kv;

        float2 y[4][MT];    // folded sums of the current tile, physical nibble pairs (0,1) (2,3) (4,5) (6,7)
        float2 acc[4][MT];  // sums of the current group since the last fold
        float sx[MT];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int t = 0; t < MT; ++t) y[q][t] = acc[q][t] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int t = 0; t < MT; ++t) sx[t] = 0.0f;

        // scales and zeros of the current group (cur) and of the next one (nxt)
        float4 sc_cur[2], zr_cur[2], sc_nxt[2], zr_nxt[2];
        sc_cur[0] = sc_cur[1] = zr_cur[0] = zr_cur[1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        sc_nxt[0] = sc_nxt[1] = zr_nxt[0] = zr_nxt[1] = sc_cur[0];
        uint32_t key_cur = 0xFFFFFFFFu, key_nxt = 0xFFFFFFFFu;  // global tile * groups + group
        uint32_t tile_cur = 0xFFFFFFFFu;
        auto load_sz = [&](uint32_t gt, uint32_t g, float4 (&sv)[2], float4 (&zv)[2]) {
            uint32_t proj, tile;
            tile_proj(a, gt, proj, tile);
            const uint32_t n = proj == 0 ? a.nq : a.nkv;
            const uint32_t wcol = tile * 32 + lane;
            sv[0] = sv[1] = zv[0] = zv[1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (wcol < n / 8) {
                const float *sc = proj == 0 ? a.sc0 : proj == 1 ? a.sc1 : a.sc2;
                const float *zr = proj == 0 ? a.zr0 : proj == 1 ? a.zr1 : a.zr2;
                const float4 *sp = reinterpret_cast<const float4 *>(sc + (size_t)g * n + 8 * wcol);
                const float4 *zp = reinterpret_cast<const float4 *>(zr + (size_t)g * n + 8 * wcol);
                sv[0] = __ldg(sp); sv[1] = __ldg(sp + 1);
                zv[0] = __ldg(zp); zv[1] = __ldg(zp + 1);
            }
        };
        // y += s (acc / 16^e - z sum x) for the rows since the last fold
        auto fold = [&]() {
            const float s8[8] = {sc_cur[0].x, sc_cur[0].y, sc_cur[0].z, sc_cur[0].w,
                                 sc_cur[1].x, sc_cur[1].y, sc_cur[1].z, sc_cur[1].w};
            const float z8[8] = {zr_cur[0].x, zr_cur[0].y, zr_cur[0].z, zr_cur[0].w,
                                 zr_cur[1].x, zr_cur[1].y, zr_cur[1].z, zr_cur[1].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int p0 = 2 * q, p1 = 2 * q + 1;
                // s / 16^e is exact: a power of two
                const float2 se = make_float2(s8[nib_col(p0)] * (1.0f / (float)(1u << (4 * nib_exp(p0)))),
                                              s8[nib_col(p1)] * (1.0f / (float)(1u << (4 * nib_exp(p1)))));
                const float2 nzs =
                    make_float2(-(z8[nib_col(p0)] * s8[nib_col(p0)]), -(z8[nib_col(p1)] * s8[nib_col(p1)]));
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    y[q][t] = __ffma2_rn(se, acc[q][t], y[q][t]);
                    y[q][t] = __ffma2_rn(nzs, make_float2(sx[t], sx[t]), y[q][t]);
                    acc[q][t] = make_float2(0.0f, 0.0f);
                }
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) sx[t] = 0.0f;
        };
        // add y into the shared totals of tile segment `seg` and clear it
        auto flush = [&](uint32_t seg) {
            float *r = red + seg * MT * kRedPitch + lane * 9;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    atomicAdd(r + t * kRedPitch + nib_col(2 * q), y[q][t].x);
                    atomicAdd(r + t * kRedPitch + nib_col(2 * q + 1), y[q][t].y);
                    y[q][t] = make_float2(0.0f, 0.0f);
                }
        };

        // position of the current half, walked forward: global tile, half
        // index within the tile (row 16 * hidx), group g and halves into it
        const uint32_t gh = a.group / 16;  // halves per group (group % 16 == 0)
        uint32_t tile_g, hidx, g, hrem;
        {
            const uint32_t hs = 2 * st_first + h_lo;  // halves from the start of tile t_first
            tile_g = t_first + hs / (2 * stages);
            hidx = hs % (2 * stages);
            g = hidx / gh;
            hrem = hidx - g * gh;
        }
        uint32_t waited = 0xFFFFFFFFu;
        for (uint32_t hu = h_lo; hu < h_hi; ++hu) {
            const uint32_t j = hu >> 1, h = hu & 1;
            const uint32_t row = 16 * hidx;  // first K row of this half
            const uint32_t cur_tile = tile_g, cur_g = g;
            // advance the walk to the next half
            if (++hrem == gh) {
                hrem = 0;
                ++g;
            }
            if (++hidx == 2 * stages) {
                hidx = 0;
                hrem = 0;
                g = 0;
                ++tile_g;
            }
            if (row >= a.k) continue;  // past K (k % 16 == 0: wholly out)
            const uint32_t key = cur_tile * a.groups + cur_g;
            if (key != key_cur) {
                if (key_cur != 0xFFFFFFFFu) {
                    fold();
                    if (cur_tile != tile_cur) flush(tile_cur - t_first);
                }
                if (key == key_nxt) {
                    sc_cur[0] = sc_nxt[0]; sc_cur[1] = sc_nxt[1];
                    zr_cur[0] = zr_nxt[0]; zr_cur[1] = zr_nxt[1];
                } else {
                    load_sz(cur_tile, cur_g, sc_cur, zr_cur);
                }
                key_cur = key;
                tile_cur = cur_tile;
                // the group after this one (next tile's first group after the
                // tile's last), loaded now so that it is in registers when needed
                const uint32_t nt = cur_g + 1 < a.groups ? cur_tile : cur_tile + 1;
                const uint32_t ng = cur_g + 1 < a.groups ? cur_g + 1 : 0;
                if (nt < tiles_total && nt <= t_first + nseg - 1) {
                    load_sz(nt, ng, sc_nxt, zr_nxt);
                    key_nxt = nt * a.groups + ng;
                } else {
                    key_nxt = 0xFFFFFFFFu;
                }
            }
            if (j != waited) {
                if (!*abort_flag && !mbar_wait(&full[j], 0, kWaitLimitNs)) fault(2);
                if (*abort_flag) break;
                waited = j;
            }
            const uint8_t *stg = smem + j * kStageS;
            const uint32_t *wp = reinterpret_cast<const uint32_t *>(stg) + 16 * h * 32 + lane;
            const float *xs = reinterpret_cast<const float *>(stg + kCodeBytes) + 16 * h;  // [MT][32], this half
            uint32_t wv[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) wv[r] = wp[r * 32];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {  // rows 4qq .. 4qq+3 of the half
                float4 xv[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    xv[t] = *reinterpret_cast<const float4 *>(xs + t * 32 + 4 * qq);
                    sx[t] += (xv[t].x + xv[t].y) + (xv[t].z + xv[t].w);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t w = wv[4 * qq + i];
                    const uint32_t hw = w >> 12;
                    const float2 f01 = __fadd2_rn(make_float2(magic_nib(w, 0xFu), magic_nib(w, 0xF0u)), kMagic);
                    const float2 f23 = __fadd2_rn(make_float2(magic_nib(w, 0xF00u), magic_nib(w, 0xF000u)), kMagic);
                    const float2 f45 = __fadd2_rn(make_float2(magic_nib(w, 0xF0000u), magic_nib(hw, 0xF00u)), kMagic);
                    const float2 f67 = __fadd2_rn(make_float2(magic_nib(hw, 0xF000u), magic_nib(hw, 0xF0000u)), kMagic);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const float xr = i == 0 ? xv[t].x : i == 1 ? xv[t].y : i == 2 ? xv[t].z : xv[t].w;
                        const float2 x2 = make_float2(xr, xr);
                        acc[0][t] = __ffma2_rn(f01, x2, acc[0][t]);
                        acc[1][t] = __ffma2_rn(f23, x2, acc[1][t]);
                        acc[2][t] = __ffma2_rn(f45, x2, acc[2][t]);
                        acc[3][t] = __ffma2_rn(f67, x2, acc[3][t]);
                    }
                }
            }
        }
        if (key_cur != 0xFFFFFFFFu && !*abort_flag) {
            fold();
            flush(tile_cur - t_first);
        }
    }

    // ---------------------------------------------------------------- drain after a timeout
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (*abort_flag) {
        if (warp == 0 && lane == 0)
            for (uint32_t j = 0; j < issued; ++j) mbar_wait(&full[j], 0, kWaitLimitNs);
        __syncthreads();
        return;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the outputs were zeroed by the previous kernel

    // ---------------------------------------------------------------- add the tiles' totals
    const uint32_t m_used = a.m < (uint32_t)MT ? a.m : (uint32_t)MT;
    for (uint32_t idx = threadIdx.x; idx < nseg * MT * 64; idx += blockDim.x) {
        const uint32_t seg = idx / (MT * 64), rest = idx % (MT * 64);  // MT * 64: a power of two
        const uint32_t t = rest / 64, quad = rest % 64;  // 4 columns: lane quad / 2, half quad % 2
        if (t >= m_used) continue;
        const uint32_t ln = quad >> 1, c0 = 4 * (quad & 1);
        uint32_t proj, tile;
        tile_proj(a, t_first + seg, proj, tile);
        const uint32_t n = proj == 0 ? a.nq : a.nkv;
        float *out = proj == 0 ? a.out0 : proj == 1 ? a.out1 : a.out2;
        const uint32_t col = tile * kColsS + 8 * ln + c0;
        if (col >= n) continue;  // n % 32 == 0: the 4 columns are all in or all out
        const float *r = red + (seg * MT + t) * kRedPitch + ln * 9 + c0;
        float *o = out + (size_t)t * n + col;
        if (vec4) {
            red_add_v4(o, r[0], r[1], r[2], r[3]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) atomicAdd(o + i, r[i]);
        }
    }
}

template <int MT>
cudaError_t launch_sk(const Int4Args &a, const CUtensorMap (&maps)[4], uint32_t vec4, cudaStream_t s) {
    using C = Sk<MT>;
    {
        static std::mutex mu;
        static std::vector<char> done;  // per device: shared-memory limit raised
        int dev = 0;
        cudaGetDevice(&dev);
        std::lock_guard<std::mutex> lock(mu);
        if ((int)done.size() <= dev) done.resize(dev + 1, 0);
        if (!done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(int4_qkv_sk_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)C::kAlloc);
            if (e != cudaSuccess) return e;
            done[dev] = 1;
        }
    }
    cudaError_t e = launch_int4_zero(a, s);
    if (e != cudaSuccess) return e;
    const uint32_t stages = (a.k + kRowsS - 1) / kRowsS;
    const uint64_t total = (uint64_t)(a.tiles_q + 2 * a.tiles_kv) * stages;
    if (total >= (1ull << 31)) return cudaErrorInvalidValue;  // unit indices are 32-bit
    // one CTA per SM; more where a range would exceed the resident stages or
    // touch more than kMaxSeg tiles (a range of L units touches at most
    // (L - 1) / stages + 2 tiles)
    uint64_t ctas = (uint64_t)device_sm_count();
    uint64_t max_len = (uint64_t)(kMaxSeg - 2) * stages + 1;
    if (max_len > (uint64_t)kMaxStages) max_len = kMaxStages;
    const uint64_t need = (total + max_len - 1) / max_len;
    if (ctas < need) ctas = need;
    if (ctas > total) ctas = total;
    if (ctas > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = QDL_TUNE_PDL ? 1 : 0;
    const uint32_t base = (uint32_t)(total / ctas), rem = (uint32_t)(total % ctas);
    return cudaLaunchKernelEx(&cfg, int4_qkv_sk_kernel<MT>, maps[0], maps[1], maps[2], maps[3], a, stages, base, rem,
                              vec4);
}

}  // namespace

bool int4_cc_supported(uint32_t nq, uint32_t nkv) { return nq % 32 == 0 && nkv % 32 == 0; }

cudaError_t launch_int4_qkv_cc(const Int4Args &a, cudaStream_t s) {
    if (a.m < 1 || a.m > 8) return cudaErrorInvalidValue;
    const uint32_t mt = a.m <= 1 ? 1 : a.m <= 2 ? 2 : a.m <= 4 ? 4 : 8;
    CUtensorMap maps[4];
    const uint32_t ns[3] = {a.nq, a.nkv, a.nkv};
    const uint32_t *qw[3] = {a.qw0, a.qw1, a.qw2};
    for (int p = 0; p < 3; ++p) {
        cudaError_t e = make_tmap_plain(&maps[p], false, qw[p], ns[p] / 8, a.k, 32, kRowsS);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = make_tmap_plain(&maps[3], true, a.x, a.k, a.m, 32, mt);
    if (e != cudaSuccess) return e;
    Int4Args b = a;  // this kernel's tiles are 256 columns wide
    b.tiles_q = (a.nq + kColsS - 1) / kColsS;
    b.tiles_kv = (a.nkv + kColsS - 1) / kColsS;
    const float *outs[3] = {a.out0, a.out1, a.out2};
    uint32_t vec4 = 1;
    for (int p = 0; p < 3; ++p) vec4 &= (reinterpret_cast<uintptr_t>(outs[p]) % 16 == 0) ? 1u : 0u;
    switch (mt) {
        case 1: return launch_sk<1>(b, maps, vec4, s);
        case 2: return launch_sk<2>(b, maps, vec4, s);
        case 4: return launch_sk<4>(b, maps, vec4, s);
        default: return launch_sk<8>(b, maps, vec4, s);
    }
}

cudaError_t read_and_clear_int4cc_fault(uint32_t *value) {
    uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_int4cc_fault, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_int4cc_fault, &zero, sizeof(uint32_t));
}

}  // namespace qdl
