// C ABI of libqdl: argument validation, dispatch and error reporting.
// Validation rules follow w8a8_decode.rs (W8a8Weight::new,
// W8a8Scratch::alloc/fits, w8a8_decode_available, w8a8_act_quant,
// w8a8_act_quant_silu, w8a8_gemv, w8a8_proj) and the shapes read by
// fused_int4_qkv.rs.  No entry point touches the device before every check
// has passed.
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "tma_pipe.cuh"

namespace qdl {

namespace {

constexpr uint32_t kWeightMagic = 0x51444C57u;  // "QDLW"
thread_local std::string g_last_error;

qdl_status fail(qdl_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

qdl_status ok() {
    g_last_error.clear();
    return QDL_OK;
}

qdl_status cuda_fail(const char *where, cudaError_t e) {
    return fail(QDL_ERR_CUDA, "%s: CUDA error %d (%s)", where, (int)e, cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_format(int32_t f) { return f == QDL_SCALE_PER_ROW || f == QDL_SCALE_BLOCK128; }

const char *format_name(int32_t f) {
    return f == QDL_SCALE_PER_ROW ? "PerRow" : (f == QDL_SCALE_BLOCK128 ? "Block128" : "invalid");
}

// W8a8Scale::act_scales_per_row
size_t scales_per_row(int32_t f, uint32_t k) { return f == QDL_SCALE_PER_ROW ? 1 : k / kKUnit; }

// W8a8Scratch::fits
bool fits(const void *q, size_t q_bytes, size_t scale_bytes, uint32_t rows, uint32_t k, int32_t f) {
    return q != nullptr && q_bytes >= (size_t)rows * k && scale_bytes >= (size_t)rows * scales_per_row(f, k) * 4;
}

qdl_status check_act_args(const char *who, int32_t format, uint32_t rows, uint32_t k, const uint8_t *q,
                          const float *q_scale, size_t q_bytes, size_t scale_bytes) {
    if (!valid_format(format)) return fail(QDL_ERR_INVALID_ARG, "%s: scale format %d is not per-row or 128x128 block", who, (int)format);
    if (rows < 1 || rows > (uint32_t)kMaxRows)
        return fail(QDL_ERR_INVALID_ARG, "%s: %u rows, want 1..=%d", who, rows, kMaxRows);
    if (k % kKUnit != 0 || k == 0 || k > QDL_MAX_K)
        return fail(QDL_ERR_INVALID_ARG, "%s: K=%u (want K %% 128 == 0, 0 < K <= %d)", who, k, QDL_MAX_K);
    if (q_scale == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: activation scale pointer is NULL", who);
    if (!fits(q, q_bytes, scale_bytes, rows, k, format))
        return fail(QDL_ERR_SCRATCH_TOO_SMALL, "%s: %u rows of K=%u do not fit the scratch", who, rows, k);
    if (!aligned(q, 16) || !aligned(q_scale, 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: q must be 16-byte and q_scale 4-byte aligned", who);
    return QDL_OK;
}

qdl_status check_input(const char *who, const char *name, const void *p, uint32_t ld, uint32_t k) {
    if (p == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: %s is NULL", who, name);
    if (ld < k || ld % 8 != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: K=%u, %s stride=%u (want K %% 128 == 0, stride >= K, stride %% 8 == 0)", who, k, name, ld);
    if (!aligned(p, 16)) return fail(QDL_ERR_INVALID_ARG, "%s: %s must be 16-byte aligned", who, name);
    return QDL_OK;
}

// The projections quantise their activations: K is bounded by what the
// quantiser covers, as for qdl_act_quant.
qdl_status check_quant_k(const char *who, uint32_t k) {
    if (k > QDL_MAX_K) return fail(QDL_ERR_INVALID_ARG, "%s: K=%u (want K %% 128 == 0, 0 < K <= %d)", who, k, QDL_MAX_K);
    return QDL_OK;
}

qdl_status check_weight(const char *who, const qdl_w8a8_weight *w) {
    if (w == nullptr || w->magic != kWeightMagic)
        return fail(QDL_ERR_INVALID_ARG, "%s: weight descriptor is NULL or was not made by qdl_w8a8_weight_init", who);
    return QDL_OK;
}

qdl_status launch_gemv(const qdl_w8a8_weight *w, const uint8_t *q, const float *q_scale, uint32_t rows, void *out,
                       int32_t out_dtype, uint32_t ldc, cudaStream_t stream, uint32_t debug_skip_iter = ~0u,
                       uint64_t wait_limit_ns = kWaitLimitNs, bool accumulate = false) {
    W8A8Args a = {};
    a.w0 = w->segs[0].weight;
    a.sw0 = w->segs[0].scale;
    a.w1 = w->count > 1 ? w->segs[1].weight : w->segs[0].weight;
    a.sw1 = w->count > 1 ? w->segs[1].scale : w->segs[0].scale;
    a.w2 = w->count > 2 ? w->segs[2].weight : w->segs[0].weight;
    a.sw2 = w->count > 2 ? w->segs[2].scale : w->segs[0].scale;
    const uint8_t *seg_w[3] = {a.w0, a.w1, a.w2};
    const uint32_t seg_n[3] = {w->segs[0].n, w->count > 1 ? w->segs[1].n : w->segs[0].n,
                               w->count > 2 ? w->segs[2].n : w->segs[0].n};
    a.q = q;
    a.sa = q_scale;
    a.out = out;
    a.m = rows;
    a.ldc = ldc;
    a.out_bf16 = out_dtype == QDL_OUT_BF16;
    a.n = w->n;
    a.k = w->k;
    a.n1 = w->n1;
    a.n2 = w->n2;
    a.kb = w->k / kKUnit;
    a.debug_skip_iter = debug_skip_iter;
    a.wait_limit_ns = wait_limit_ns;
    a.accumulate = out_dtype == QDL_OUT_F32_ADD || (accumulate && out_dtype == QDL_OUT_F32);
    a.out_zeroed = accumulate && out_dtype == QDL_OUT_F32;
    // one pass of the tcgen05 kernel for any rows <= 256
    cudaError_t e = launch_w8a8_gemm_tc(a, w->format, seg_w, seg_n, stream);
    if (e != cudaSuccess) return cuda_fail("qdl_w8a8_gemv", e);
    return ok();
}

// split-K factor the tcgen05 GEMV takes for this weight and row count when
// its ranks add into a zeroed f32 output (as the projection runs it)
uint32_t gemv_split(const qdl_w8a8_weight *w, uint32_t rows) {
    W8A8Args a = {};
    a.accumulate = 1;
    a.n = w->n;
    a.k = w->k;
    a.kb = w->k / kKUnit;
    a.m = rows;
    PlanInfo p = {};
    return plan_w8a8_gemm_tc(a, w->format, &p) == cudaSuccess ? p.split : 1;
}

// The projection entry points with f32 output let the quantiser zero the
// output first, so that the GEMV's split-K ranks add into it atomically
// instead of meeting in a cluster reduction.
bool proj_accumulates(const qdl_w8a8_weight *w, uint32_t rows) {
    return gemv_split(w, rows) >= 2 || w8a8_streamk_applies(w->format, rows);
}

bool zero_f32_output(ActQuantArgs &a, const qdl_w8a8_weight *w, uint32_t rows, void *out, int32_t out_dtype,
                     uint32_t ldc, uint32_t n) {
    if (out_dtype != QDL_OUT_F32 || !proj_accumulates(w, rows)) return false;
    a.zout = static_cast<float *>(out);
    a.zldc = ldc;
    a.zn = n;
    return true;
}

}  // namespace

int device_sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace qdl

using namespace qdl;

extern "C" {

const char *qdl_last_error(void) { return g_last_error.c_str(); }

const char *qdl_status_string(qdl_status s) {
    switch (s) {
        case QDL_OK: return "QDL_OK";
        case QDL_ERR_INVALID_ARG: return "QDL_ERR_INVALID_ARG";
        case QDL_ERR_SCRATCH_TOO_SMALL: return "QDL_ERR_SCRATCH_TOO_SMALL";
        case QDL_ERR_UNSUPPORTED: return "QDL_ERR_UNSUPPORTED";
        case QDL_ERR_CUDA: return "QDL_ERR_CUDA";
        case QDL_ERR_DEVICE_TIMEOUT: return "QDL_ERR_DEVICE_TIMEOUT";
    }
    return "QDL_ERR_UNKNOWN";
}

qdl_status qdl_w8a8_weight_init(qdl_w8a8_weight *out, const qdl_fp8_segment *segs, uint32_t count) {
    const char *who = "W8a8Weight";
    if (out == nullptr || segs == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: NULL descriptor or segment list", who);
    if (count < 1 || count > 3) return fail(QDL_ERR_INVALID_ARG, "%s: %u segments, want 1..=3", who, count);
    const int32_t format = segs[0].format;
    if (!valid_format(format))
        return fail(QDL_ERR_INVALID_ARG, "%s: scale format %d is not per-row or 128x128 block", who, (int)format);
    const uint32_t k = segs[0].k;
    if (k == 0 || k % kKUnit != 0) return fail(QDL_ERR_INVALID_ARG, "%s: K=%u is not a positive multiple of %d", who, k, kKUnit);
    const uint32_t align = format == QDL_SCALE_PER_ROW ? 16 : 128;  // W8a8Scale::segment_align
    uint64_t total = 0;
    for (uint32_t i = 0; i < count; ++i) {
        const qdl_fp8_segment &s = segs[i];
        if (s.k != k || s.format != format)
            return fail(QDL_ERR_INVALID_ARG, "%s: segment %u is [%u, %u] %s, segment 0 is [.., %u] %s", who, i, s.n, s.k,
                        format_name(s.format), k, format_name(format));
        if (s.n == 0 || s.weight == nullptr || s.scale == nullptr)
            return fail(QDL_ERR_INVALID_ARG, "%s: segment %u is empty", who, i);
        if (i + 1 < count && s.n % align != 0)
            return fail(QDL_ERR_INVALID_ARG, "%s: segment %u has %u rows, not a multiple of %u", who, i, s.n, align);
        if (!aligned(s.weight, 16) || !aligned(s.scale, 4))
            return fail(QDL_ERR_INVALID_ARG, "%s: segment %u weight must be 16-byte and scale 4-byte aligned", who, i);
        total += s.n;
    }
    if (total >= (1ull << 31)) return fail(QDL_ERR_UNSUPPORTED, "%s: total N=%llu exceeds 2^31", who, (unsigned long long)total);
    qdl_w8a8_weight w = {};
    for (uint32_t i = 0; i < 3; ++i) w.segs[i] = segs[i < count ? i : 0];
    w.count = count;
    w.n = (uint32_t)total;
    w.k = k;
    w.format = format;
    // W8a8Weight::boundaries
    const uint32_t n0 = segs[0].n;
    w.n1 = count == 1 ? w.n : n0;
    w.n2 = count == 3 ? n0 + segs[1].n : w.n;
    w.magic = kWeightMagic;
    *out = w;
    return ok();
}

qdl_status qdl_scratch_bytes(uint32_t max_k, size_t *q_bytes, size_t *scale_bytes) {
    const size_t rows = kMaxRows;
    const size_t groups = ((size_t)max_k + kKUnit - 1) / kKUnit;  // no 32-bit wrap near UINT32_MAX
    if (q_bytes) *q_bytes = rows * max_k;
    if (scale_bytes) *scale_bytes = rows * (groups > 1 ? groups : 1) * 4;
    return ok();
}

qdl_status qdl_act_quant(int32_t format, const void *x, uint32_t ldx, uint32_t rows, uint32_t k, uint8_t *q, float *q_scale,
                         size_t q_bytes, size_t scale_bytes, void *stream) {
    const char *who = "w8a8_act_quant";
    qdl_status st = check_act_args(who, format, rows, k, q, q_scale, q_bytes, scale_bytes);
    if (st != QDL_OK) return st;
    if ((st = check_input(who, "x", x, ldx, k)) != QDL_OK) return st;
    ActQuantArgs a = {static_cast<const uint16_t *>(x), nullptr, ldx, 0, rows, k, q, q_scale};
    cudaError_t e = launch_act_quant(a, format, false, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(who, e);
    return ok();
}

qdl_status qdl_act_quant_silu(int32_t format, const void *gate, const void *up, uint32_t ld_gate, uint32_t ld_up, uint32_t rows,
                              uint32_t k, uint8_t *q, float *q_scale, size_t q_bytes, size_t scale_bytes, void *stream) {
    const char *who = "w8a8_act_quant_silu";
    qdl_status st = check_act_args(who, format, rows, k, q, q_scale, q_bytes, scale_bytes);
    if (st != QDL_OK) return st;
    if ((st = check_input(who, "gate", gate, ld_gate, k)) != QDL_OK) return st;
    if ((st = check_input(who, "up", up, ld_up, k)) != QDL_OK) return st;
    ActQuantArgs a = {static_cast<const uint16_t *>(gate), static_cast<const uint16_t *>(up), ld_gate, ld_up, rows, k, q, q_scale};
    cudaError_t e = launch_act_quant(a, format, true, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(who, e);
    return ok();
}

static qdl_status check_gemv(const char *who, const qdl_w8a8_weight *w, const uint8_t *q, const float *q_scale, size_t q_bytes,
                             size_t scale_bytes, uint32_t rows, const void *out, int32_t out_dtype, uint32_t ldc, bool allow_add = false,
                             uint32_t max_rows = kMaxRows) {
    qdl_status st = check_weight(who, w);
    if (st != QDL_OK) return st;
    // w8a8_decode_available; more than 256 rows (projections only) run in
    // passes of 256 rows through the same scratch
    const uint32_t pass_rows = rows < (uint32_t)kMaxRows ? rows : (uint32_t)kMaxRows;
    if (rows < 1 || rows > max_rows || q_scale == nullptr || !fits(q, q_bytes, scale_bytes, pass_rows, w->k, w->format))
        return fail(rows < 1 || rows > max_rows || q_scale == nullptr ? QDL_ERR_INVALID_ARG : QDL_ERR_SCRATCH_TOO_SMALL,
                    "%s: not available for %u rows of [%u, %u] %s", who, rows, w->n, w->k, format_name(w->format));
    if (!aligned(q, 16) || !aligned(q_scale, 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: q must be 16-byte and q_scale 4-byte aligned", who);
    if (ldc < w->n) return fail(QDL_ERR_INVALID_ARG, "%s: ldc=%u < N=%u", who, ldc, w->n);
    if (out_dtype != QDL_OUT_F32 && out_dtype != QDL_OUT_BF16 && out_dtype != QDL_OUT_F32_DETERMINISTIC &&
        !(allow_add && out_dtype == QDL_OUT_F32_ADD))
        return fail(QDL_ERR_INVALID_ARG, "%s: output dtype %d is not %s", who, (int)out_dtype,
                    allow_add ? "F32, BF16, F32_ADD or F32_DETERMINISTIC" : "F32, BF16 or F32_DETERMINISTIC");
    if (out == nullptr || !aligned(out, out_dtype == QDL_OUT_BF16 ? 2 : 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: output is NULL or misaligned", who);
    return QDL_OK;
}

qdl_status qdl_w8a8_gemv(const qdl_w8a8_weight *w, const uint8_t *q, const float *q_scale, size_t q_bytes, size_t scale_bytes,
                         uint32_t rows, void *out, int32_t out_dtype, uint32_t ldc, void *stream) {
    qdl_status st = check_gemv("w8a8_gemv", w, q, q_scale, q_bytes, scale_bytes, rows, out, out_dtype, ldc, true);
    if (st != QDL_OK) return st;
    return launch_gemv(w, q, q_scale, rows, out, out_dtype, ldc, static_cast<cudaStream_t>(stream));
}

namespace {

// One decode projection of up to 256 rows: the quantiser (plain or SiLU),
// then the GEMV.
qdl_status proj_pass(const char *who, const qdl_w8a8_weight *w, const void *x, const void *up, uint32_t ldx, uint32_t ld_up,
                     bool silu, uint32_t rows, void *out, int32_t out_dtype, uint32_t ldc, uint8_t *q, float *q_scale,
                     cudaStream_t stream) {
    ActQuantArgs a = {static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(up), ldx, ld_up, rows, w->k, q, q_scale};
    const bool acc = zero_f32_output(a, w, rows, out, out_dtype, ldc, w->n);
    cudaError_t e = launch_act_quant(a, w->format, silu, stream);
    if (e != cudaSuccess) return cuda_fail(who, e);
    return launch_gemv(w, q, q_scale, rows, out, out_dtype, ldc, stream, ~0u, kWaitLimitNs, acc);
}

// Rows beyond 256 (a prefill-shaped call).  When the scratch holds every
// row, the rows are quantised 256 at a time into their own parts of it and
// one GEMV launch covers them all: its token blocks of one weight tile run
// side by side, so the weights stream from HBM once.  Otherwise the call runs
// in passes of 256 rows, in order on the stream: each pass quantises into the
// same scratch, which the next pass's quantiser overwrites only after the
// previous GEMV has finished (programmatic launch orders every library kernel
// after its predecessor), and each pass streams the weights again.
qdl_status proj_passes(const char *who, const qdl_w8a8_weight *w, const void *x, const void *up, uint32_t ldx, uint32_t ld_up,
                       bool silu, uint32_t rows, void *out, int32_t out_dtype, uint32_t ldc, uint8_t *q, float *q_scale,
                       size_t q_bytes, size_t scale_bytes, void *stream) {
    const size_t elt = out_dtype == QDL_OUT_BF16 ? 2 : 4;
    if (rows > (uint32_t)kMaxRows && fits(q, q_bytes, scale_bytes, rows, w->k, w->format)) {
        const cudaStream_t s = static_cast<cudaStream_t>(stream);
        const size_t spr = scales_per_row(w->format, w->k);
        const bool acc = out_dtype == QDL_OUT_F32 && proj_accumulates(w, rows);
        for (uint32_t done = 0; done < rows; done += (uint32_t)kMaxRows) {
            const uint32_t n = rows - done < (uint32_t)kMaxRows ? rows - done : (uint32_t)kMaxRows;
            ActQuantArgs a = {static_cast<const uint16_t *>(x) + (size_t)done * ldx,
                              silu ? static_cast<const uint16_t *>(up) + (size_t)done * ld_up : nullptr,
                              ldx, ld_up, n, w->k, q + (size_t)done * w->k, q_scale + (size_t)done * spr};
            if (acc) {  // this chunk's quantiser zeroes its rows of the output
                a.zout = reinterpret_cast<float *>(static_cast<uint8_t *>(out) + (size_t)done * ldc * elt);
                a.zldc = ldc;
                a.zn = w->n;
            }
            cudaError_t e = launch_act_quant(a, w->format, silu, s);
            if (e != cudaSuccess) return cuda_fail(who, e);
        }
        return launch_gemv(w, q, q_scale, rows, out, out_dtype, ldc, s, ~0u, kWaitLimitNs, acc);
    }
    for (uint32_t done = 0; done < rows; done += (uint32_t)kMaxRows) {
        const uint32_t n = rows - done < (uint32_t)kMaxRows ? rows - done : (uint32_t)kMaxRows;
        const uint16_t *xp = static_cast<const uint16_t *>(x) + (size_t)done * ldx;
        const uint16_t *up_p = silu ? static_cast<const uint16_t *>(up) + (size_t)done * ld_up : nullptr;
        void *op = static_cast<uint8_t *>(out) + (size_t)done * ldc * elt;
        qdl_status st = proj_pass(who, w, xp, up_p, ldx, ld_up, silu, n, op, out_dtype, ldc, q, q_scale,
                                  static_cast<cudaStream_t>(stream));
        if (st != QDL_OK) return st;
    }
    return ok();
}

}  // namespace

qdl_status qdl_w8a8_proj(const qdl_w8a8_weight *w, const void *x, uint32_t ldx, uint32_t rows, void *out, int32_t out_dtype,
                         uint32_t ldc, uint8_t *q, float *q_scale, size_t q_bytes, size_t scale_bytes, void *stream) {
    const char *who = "w8a8_proj";
    qdl_status st = check_gemv(who, w, q, q_scale, q_bytes, scale_bytes, rows, out, out_dtype, ldc, false, QDL_MAX_PROJ_ROWS);
    if (st != QDL_OK) return st;
    if ((st = check_quant_k(who, w->k)) != QDL_OK) return st;
    if ((st = check_input(who, "x", x, ldx, w->k)) != QDL_OK) return st;
    return proj_passes(who, w, x, nullptr, ldx, 0, false, rows, out, out_dtype, ldc, q, q_scale, q_bytes, scale_bytes,
                       stream);
}

qdl_status qdl_w8a8_proj_silu(const qdl_w8a8_weight *w, const void *gate, const void *up, uint32_t ld_gate, uint32_t ld_up,
                              uint32_t rows, void *out, int32_t out_dtype, uint32_t ldc, uint8_t *q, float *q_scale, size_t q_bytes,
                              size_t scale_bytes, void *stream) {
    const char *who = "w8a8_proj_silu";
    qdl_status st = check_gemv(who, w, q, q_scale, q_bytes, scale_bytes, rows, out, out_dtype, ldc, false, QDL_MAX_PROJ_ROWS);
    if (st != QDL_OK) return st;
    if ((st = check_quant_k(who, w->k)) != QDL_OK) return st;
    if ((st = check_input(who, "gate", gate, ld_gate, w->k)) != QDL_OK) return st;
    if ((st = check_input(who, "up", up, ld_up, w->k)) != QDL_OK) return st;
    return proj_passes(who, w, gate, up, ld_gate, ld_up, true, rows, out, out_dtype, ldc, q, q_scale, q_bytes, scale_bytes,
                       stream);
}

qdl_status qdl_int4_qkv_gemv(const float *x, uint32_t m, uint32_t k, uint32_t nq, uint32_t nkv, uint32_t group,
                             const uint32_t *const *qw, const float *const *sc, const float *const *zr, float *const *out,
                             void *stream) {
    const char *who = "fused_int4_qkv";
    if (x == nullptr || qw == nullptr || sc == nullptr || zr == nullptr || out == nullptr)
        return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (m < 1) return fail(QDL_ERR_INVALID_ARG, "%s: m=%u, want m >= 1", who, m);
    if (group == 0 || group % 16 != 0 || k == 0 || k % group != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: k=%u, group=%u (want group > 0, group %% 16 == 0, k %% group == 0)", who, k, group);
    if (nq == 0 || nkv == 0 || nq % 8 != 0 || nkv % 8 != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: nq=%u, nkv=%u (want positive multiples of 8)", who, nq, nkv);
    if (!aligned(x, 16)) return fail(QDL_ERR_INVALID_ARG, "%s: x must be 16-byte aligned", who);
    bool vec2 = nq % 16 == 0 && nkv % 16 == 0;
    bool qw16 = true;  // the TMA kernels stream codes from 16-byte aligned bases
    for (int p = 0; p < 3; ++p) {
        if (qw[p] == nullptr || sc[p] == nullptr || zr[p] == nullptr || out[p] == nullptr)
            return fail(QDL_ERR_INVALID_ARG, "%s: projection %d has a NULL pointer", who, p);
        if (!aligned(qw[p], 4) || !aligned(sc[p], 16) || !aligned(zr[p], 16) || !aligned(out[p], 4))
            return fail(QDL_ERR_INVALID_ARG, "%s: projection %d misaligned (qw 4, sc/zr 16, out 4 bytes)", who, p);
        vec2 = vec2 && aligned(qw[p], 8);
        qw16 = qw16 && aligned(qw[p], 16);
    }
    Int4Args a = {};
    a.qw0 = qw[0]; a.qw1 = qw[1]; a.qw2 = qw[2];
    a.sc0 = sc[0]; a.sc1 = sc[1]; a.sc2 = sc[2];
    a.zr0 = zr[0]; a.zr1 = zr[1]; a.zr2 = zr[2];
    a.k = k;
    a.group = group;
    a.groups = k / group;
    a.nq = nq;
    a.nkv = nkv;
    a.tiles_q = (nq + 127) / 128;
    a.tiles_kv = (nkv + 127) / 128;
    a.vec2 = vec2;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // widths multiples of 32: the CUDA-core stream-K kernel for up to
    // QDL_INT4_CC_MAX_ROWS rows (up to 8 where the tcgen05 kernel does not
    // apply); above that, group 128: the tcgen05 kernel, QDL_INT4_TC_PASS_ROWS
    // rows per pass;
    // otherwise the mma.sync kernel, 16 rows per pass
    const bool tc = qw16 && int4_tc_supported(nq, nkv, group);
    static_assert(QDL_INT4_CC_MAX_ROWS <= 8, "the CUDA-core kernel takes up to 8 rows");
    if (qw16 && int4_cc_supported(nq, nkv) && (m <= QDL_INT4_CC_MAX_ROWS || (m <= 8 && !tc))) {
        a.x = x;
        a.out0 = out[0];
        a.out1 = out[1];
        a.out2 = out[2];
        a.m = m;
        cudaError_t e = launch_int4_qkv_cc(a, s);
        if (e != cudaSuccess) return cuda_fail(who, e);
        return ok();
    }
    static_assert(QDL_INT4_TC_PASS_ROWS == 16 || QDL_INT4_TC_PASS_ROWS == 32, "tcgen05 AWQ passes of 16 or 32 rows");
    const uint32_t chunk = tc ? QDL_INT4_TC_PASS_ROWS : 16;
    for (uint32_t done = 0; done < m; done += chunk) {
        const uint32_t mm = m - done < chunk ? m - done : chunk;
        a.x = x + (size_t)done * k;
        a.out0 = out[0] + (size_t)done * nq;
        a.out1 = out[1] + (size_t)done * nkv;
        a.out2 = out[2] + (size_t)done * nkv;
        a.m = mm;
        cudaError_t e = tc ? launch_int4_qkv_tc(a, s) : launch_int4_qkv(a, s);
        if (e != cudaSuccess) return cuda_fail(who, e);
    }
    return ok();
}

// ---------------------------------------------------------------- KV-cache quantisers
//
// kv_cache_quant.wgsl.  Shapes: x and out [tokens, head_dim] f32; int8 codes
// [tokens, head_dim] with scales [tokens]; INT4 over the flattened
// tokens * head_dim values, packed two per byte, scales and zeros
// [tokens * head_dim / group].

namespace {

qdl_status check_kv_shape(const char *who, uint32_t tokens, uint32_t head_dim) {
    if (tokens < 1 || head_dim < 1 || head_dim % 4 != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: tokens=%u, head_dim=%u (want tokens >= 1, head_dim a positive multiple of 4)",
                    who, tokens, head_dim);
    if ((uint64_t)tokens * head_dim >= (1ull << 31))
        return fail(QDL_ERR_UNSUPPORTED, "%s: tokens * head_dim = %llu exceeds 2^31", who,
                    (unsigned long long)tokens * head_dim);
    return QDL_OK;
}

qdl_status check_kv_int4(const char *who, uint32_t tokens, uint32_t head_dim, uint32_t group) {
    qdl_status st = check_kv_shape(who, tokens, head_dim);
    if (st != QDL_OK) return st;
    if (group == 0 || group % 8 != 0 || ((uint64_t)tokens * head_dim) % group != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: group=%u (want a positive multiple of 8 dividing tokens * head_dim = %llu)",
                    who, group, (unsigned long long)tokens * head_dim);
    return QDL_OK;
}

}  // namespace

// ---------------------------------------------------------------- weight preparation

qdl_status qdl_fp8_weight_quant(int32_t format, const void *w, int32_t w_dtype, uint32_t ldw, uint32_t n, uint32_t k,
                                uint8_t *codes, float *scales, void *stream) {
    const char *who = "qdl_fp8_weight_quant";
    if (format != QDL_SCALE_PER_ROW && format != QDL_SCALE_BLOCK128)
        return fail(QDL_ERR_INVALID_ARG, "%s: format=%d is not PER_ROW or BLOCK128", who, format);
    if (w_dtype != QDL_IN_F32 && w_dtype != QDL_IN_BF16)
        return fail(QDL_ERR_INVALID_ARG, "%s: w_dtype=%d is not F32 or BF16", who, w_dtype);
    if (n < 1 || k < 128 || k % 128 != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: n=%u, k=%u (want n >= 1, k a positive multiple of 128)", who, n, k);
    const uint32_t lda = w_dtype == QDL_IN_BF16 ? 8 : 4;
    if (ldw < k || ldw % lda != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: ldw=%u (want ldw >= k and a multiple of %u)", who, ldw, lda);
    if (w == nullptr || codes == nullptr || scales == nullptr)
        return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned(w, 16) || !aligned(codes, 8) || !aligned(scales, 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: w must be 16-byte, codes 8-byte, scales 4-byte aligned", who);
    if (format == QDL_SCALE_PER_ROW && n > 0x7FFFFFFFu)
        return fail(QDL_ERR_UNSUPPORTED, "%s: n=%u rows exceed the grid", who, n);
    cudaError_t e = launch_fp8_weight_quant(format, w, w_dtype == QDL_IN_BF16, ldw, n, k, codes, scales,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(who, e);
}

qdl_status qdl_awq_pack(const uint8_t *nib, uint32_t k, uint32_t n, uint32_t *qw, void *stream) {
    const char *who = "qdl_awq_pack";
    if (k < 1 || n < 8 || n % 8 != 0)
        return fail(QDL_ERR_INVALID_ARG, "%s: k=%u, n=%u (want k >= 1, n a positive multiple of 8)", who, k, n);
    if (nib == nullptr || qw == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned(nib, 8) || !aligned(qw, 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: nib must be 8-byte, qw 4-byte aligned", who);
    cudaError_t e = launch_awq_pack(nib, k, n, qw, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(who, e);
}

// ---------------------------------------------------------------- KV-cache codecs (entry points)

qdl_status qdl_kv_quant_int8(const float *x, uint32_t tokens, uint32_t head_dim, int8_t *q, float *scale,
                             void *stream) {
    const char *who = "quantize_kv_int8";
    qdl_status st = check_kv_shape(who, tokens, head_dim);
    if (st != QDL_OK) return st;
    if (x == nullptr || q == nullptr || scale == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned(x, 16) || !aligned(q, 4) || !aligned(scale, 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: x must be 16-byte, q and scale 4-byte aligned", who);
    cudaError_t e = launch_kv_quant_int8(x, tokens, head_dim, q, scale, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(who, e);
}

qdl_status qdl_kv_dequant_int8(const int8_t *q, const float *scale, uint32_t tokens, uint32_t head_dim, float *out,
                               void *stream) {
    const char *who = "dequantize_kv_int8";
    qdl_status st = check_kv_shape(who, tokens, head_dim);
    if (st != QDL_OK) return st;
    if (q == nullptr || scale == nullptr || out == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned(q, 4) || !aligned(scale, 4) || !aligned(out, 16))
        return fail(QDL_ERR_INVALID_ARG, "%s: q and scale must be 4-byte, out 16-byte aligned", who);
    cudaError_t e = launch_kv_dequant_int8(q, scale, tokens, head_dim, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(who, e);
}

qdl_status qdl_kv_quant_int4(const float *x, uint32_t tokens, uint32_t head_dim, uint32_t group, uint8_t *packed,
                             float *scale, float *zero, void *stream) {
    const char *who = "quantize_kv_int4";
    qdl_status st = check_kv_int4(who, tokens, head_dim, group);
    if (st != QDL_OK) return st;
    if (x == nullptr || packed == nullptr || scale == nullptr || zero == nullptr)
        return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned(x, 16) || !aligned(packed, 4) || !aligned(scale, 4) || !aligned(zero, 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: x must be 16-byte, packed, scale and zero 4-byte aligned", who);
    cudaError_t e = launch_kv_quant_int4(x, (size_t)tokens * head_dim, group, packed, scale, zero,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(who, e);
}

qdl_status qdl_kv_dequant_int4(const uint8_t *packed, const float *scale, const float *zero, uint32_t tokens,
                               uint32_t head_dim, uint32_t group, float *out, void *stream) {
    const char *who = "dequantize_kv_int4";
    qdl_status st = check_kv_int4(who, tokens, head_dim, group);
    if (st != QDL_OK) return st;
    if (packed == nullptr || scale == nullptr || zero == nullptr || out == nullptr)
        return fail(QDL_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned(packed, 4) || !aligned(scale, 4) || !aligned(zero, 4) || !aligned(out, 16))
        return fail(QDL_ERR_INVALID_ARG, "%s: packed, scale and zero must be 4-byte, out 16-byte aligned", who);
    cudaError_t e = launch_kv_dequant_int4(packed, scale, zero, (size_t)tokens * head_dim, group, out,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(who, e);
}

// ---------------------------------------------------------------- no-allocation variant
//
// qdl_w8a8_proj_static: the decode projection for callers that cannot
// allocate device memory.  Its activation codes and scales live in the
// fixed device array below instead of caller scratch.  The array's host-side
// name is only a stand-in for the symbol; the device address is looked up
// once per device (cudaGetSymbolAddress, on the first call made with that
// device current) and then passed to the kernels like any scratch pointer.

static __device__ __align__(256) uint8_t g_static_scratch[QDL_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_static_mu;
std::vector<void *> g_static_addr;  // per device; nullptr until looked up

qdl_status static_scratch_address(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("w8a8_proj_static", e);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if ((int)g_static_addr.size() <= dev) g_static_addr.resize(dev + 1, nullptr);
    if (g_static_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) return cuda_fail("w8a8_proj_static: cudaGetSymbolAddress", e);
        g_static_addr[dev] = p;
    }
    *addr = g_static_addr[dev];
    return QDL_OK;
}

}  // namespace

qdl_status qdl_w8a8_proj_static(const qdl_w8a8_weight *w, const void *x, uint32_t ldx, uint32_t rows, void *out,
                                int32_t out_dtype, uint32_t ldc, void *stream) {
    const char *who = "w8a8_proj_static";
    qdl_status st = check_weight(who, w);
    if (st != QDL_OK) return st;
    if (rows < 1 || rows > (uint32_t)kMaxRows) return fail(QDL_ERR_INVALID_ARG, "%s: %u rows, want 1..=%d", who, rows, kMaxRows);
    if ((st = check_quant_k(who, w->k)) != QDL_OK) return st;
    const size_t q_bytes = (size_t)rows * w->k;
    const size_t scale_off = (q_bytes + 255) / 256 * 256;
    const size_t scale_bytes = (size_t)rows * scales_per_row(w->format, w->k) * 4;
    if (scale_off + scale_bytes > (size_t)QDL_STATIC_SCRATCH_BYTES)
        return fail(QDL_ERR_UNSUPPORTED, "%s: %u rows of K=%u need %zu bytes of static scratch, the limit is %d", who, rows,
                    w->k, scale_off + scale_bytes, QDL_STATIC_SCRATCH_BYTES);
    if (ldc < w->n) return fail(QDL_ERR_INVALID_ARG, "%s: ldc=%u < N=%u", who, ldc, w->n);
    if (out_dtype != QDL_OUT_F32 && out_dtype != QDL_OUT_BF16 && out_dtype != QDL_OUT_F32_DETERMINISTIC)
        return fail(QDL_ERR_INVALID_ARG, "%s: output dtype %d is not F32, BF16 or F32_DETERMINISTIC", who,
                    (int)out_dtype);
    if (out == nullptr || !aligned(out, out_dtype == QDL_OUT_BF16 ? 2 : 4))
        return fail(QDL_ERR_INVALID_ARG, "%s: output is NULL or misaligned", who);
    if ((st = check_input(who, "x", x, ldx, w->k)) != QDL_OK) return st;
    void *base = nullptr;
    if ((st = static_scratch_address(&base)) != QDL_OK) return st;
    uint8_t *q = static_cast<uint8_t *>(base);
    float *q_scale = reinterpret_cast<float *>(static_cast<uint8_t *>(base) + scale_off);
    // every code and scale the GEMV reads is written by the quantiser first,
    // so nothing left over from an earlier call is ever read
    ActQuantArgs a = {static_cast<const uint16_t *>(x), nullptr, ldx, 0, rows, w->k, q, q_scale};
    cudaError_t e = launch_act_quant(a, w->format, false, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(who, e);
    return launch_gemv(w, q, q_scale, rows, out, out_dtype, ldc, static_cast<cudaStream_t>(stream));
}

qdl_status qdl_w8a8_plan(const qdl_w8a8_weight *w, uint32_t rows, qdl_plan *plan) {
    const char *who = "w8a8_plan";
    qdl_status st = check_weight(who, w);
    if (st != QDL_OK) return st;
    if (plan == nullptr) return fail(QDL_ERR_INVALID_ARG, "%s: plan is NULL", who);
    if (rows < 1 || rows > (uint32_t)kMaxRows) return fail(QDL_ERR_INVALID_ARG, "%s: %u rows, want 1..=%d", who, rows, kMaxRows);
    W8A8Args a = {};
    a.n = w->n;
    a.k = w->k;
    a.kb = w->k / kKUnit;
    a.m = rows;
    PlanInfo p = {};
    cudaError_t e = plan_w8a8_gemm_tc(a, w->format, &p);
    if (e != cudaSuccess) return cuda_fail(who, e);
    plan->kernel = p.kernel;
    plan->mma_n = p.mma_n;
    plan->tiles = p.tiles;
    plan->split_k = p.split;
    plan->stages = p.stages;
    plan->threads = p.threads;
    plan->smem_bytes = p.smem;
    plan->resident_clusters = p.clusters;
    plan->proj_launches = 2u;  // the quantiser, then the GEMV
    plan->proj_accumulates = proj_accumulates(w, rows) ? 1u : 0u;
    plan->proj_streamk = plan->proj_accumulates && w8a8_streamk_applies(w->format, rows) ? 1u : 0u;
    return ok();
}

qdl_status qdl_check_device_fault(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("qdl_check_device_fault", e);
    uint32_t word = 0, word_tc = 0;
    if ((e = read_and_clear_tc_fault(&word)) != cudaSuccess) return cuda_fail("qdl_check_device_fault", e);
    if ((e = read_and_clear_int4_fault(&word_tc)) != cudaSuccess) return cuda_fail("qdl_check_device_fault", e);
    word |= word_tc;
    if ((e = read_and_clear_int4cc_fault(&word_tc)) != cudaSuccess) return cuda_fail("qdl_check_device_fault", e);
    word |= word_tc;
    if (word != 0)
        return fail(QDL_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (fault word 0x%x: 1 = producer, 2/8 = consumer or MMA, 4/16/32 = accumulator)",
                    word);
    return ok();
}

qdl_status qdl_selftest_bounded_wait(const qdl_w8a8_weight *w, const uint8_t *q, const float *q_scale, size_t q_bytes,
                                     size_t scale_bytes, uint32_t rows, float *out, uint32_t limit_us, void *stream) {
    const char *who = "selftest_bounded_wait";
    qdl_status st = check_gemv(who, w, q, q_scale, q_bytes, scale_bytes, rows, out, QDL_OUT_F32, w ? w->n : 0);
    if (st != QDL_OK) return st;
    if (limit_us == 0 || limit_us > 1000000) return fail(QDL_ERR_INVALID_ARG, "%s: limit_us=%u, want 1..1000000", who, limit_us);
    st = launch_gemv(w, q, q_scale, rows, out, QDL_OUT_F32, w->n, static_cast<cudaStream_t>(stream), 0,
                     (uint64_t)limit_us * 1000ull);
    if (st != QDL_OK) return st;
    return qdl_check_device_fault(stream);
}

}  // extern "C"
