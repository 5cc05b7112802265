/*
 * qdl oracle: plain, slow CPU reference.  TEST INFRASTRUCTURE ONLY (see
 * qdl_oracle.h).  Build with -ffp-contract=off so that every float
 * operation below is one IEEE-754 binary32 operation rounded to nearest:
 * the activation codes must come out bit-exact, so the order and rounding
 * of each step is part of the definition.
 */
#include "qdl_oracle.h"

#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

static void *malloc_or_die(size_t bytes) {
    void *p = malloc(bytes ? bytes : 1);
    if (!p) {
        fprintf(stderr, "qdl oracle: out of host memory (%zu bytes)\n", bytes);
        abort();
    }
    return p;
}

static float bits_to_f32(uint32_t b) {
    float f;
    memcpy(&f, &b, 4);
    return f;
}

static float bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* ---------------------------------------------------------------------
 * FP8 E4M3 (OCP OFP8 specification, "E4M3" format).
 *   sign | 4-bit exponent, bias 7 | 3-bit mantissa
 *   exponent field 0      : subnormal, value = m * 2^-9        (m = 1..7)
 *   exponent field 1..15  : normal,    value = (1 + m/8) * 2^(e-7)
 *   S.1111.111            : NaN (so the largest finite value is 448)
 * No infinities.
 * ------------------------------------------------------------------- */

float orc_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return (float)(sign ? -mag : mag);
}

/* round a non-negative double holding an exact multiple of 2^-40 or so to
 * the nearest integer, ties to even */
static double round_half_even(double q) {
    double fl = floor(q);
    double d = q - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Nearest E4M3 value, ties to the even mantissa, magnitudes beyond the
 * largest finite value saturate to +-448 ("satfinite").  -0 keeps its
 * sign.  NaN input is outside the contract. */
uint8_t orc_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v); /* exact */
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid, step 2^-9; a result of 8 steps is 2^-6, which is
         * the code 0x08 (exponent field 1, mantissa 0): the encoding is
         * continuous across the boundary. */
        double q = round_half_even(a / ldexp(1.0, -9));
        return sign | (uint8_t)q;
    }
    int e2;
    frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1; /* a in [2^E, 2^(E+1)) */
    double step = ldexp(1.0, E - 3);
    double q = round_half_even(a / step); /* 8..16 */
    if (q == 16.0) {
        E += 1;
        q = 8.0;
    }
    /* a < 448 keeps E <= 8 and, at E == 8, q <= 14 (448 itself). */
    return sign | (uint8_t)(((E + 7) << 3) | ((int)q - 8));
}

void orc_e4m3_encode_n(const float *v, size_t n, uint8_t *out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_decode_n(const uint8_t *c, size_t n, float *out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}

/* ---------------------------------------------------------------------
 * qdl exp: the library's own written specification of exp in binary32,
 * built only from correctly rounded add/mul/fma and exact scaling by 2^n,
 * so that any two conforming implementations agree bit for bit.
 * Method: Cody and Waite argument reduction, x = n ln2 + r with
 * n = rint(x log2 e) and ln2 split into a binary32 head and tail, then the
 * degree-7 Taylor polynomial of e^r (coefficients 1/j! rounded to binary32)
 * in Horner form, then multiplication by 2^n.
 * ------------------------------------------------------------------- */

#define ORC_EXP_HI 0x42b17218u    /* 88.72284f  = RN32(ln FLT_MAX)      */
#define ORC_EXP_LO 0xc2cff1b4u    /* -103.97208f = RN32(ln 2^-150)      */
#define ORC_LOG2E 0x3fb8aa3bu     /* RN32(1/ln 2)                       */
#define ORC_LN2_HEAD 0x3f317218u  /* RN32(ln 2)                         */
#define ORC_LN2_TAIL 0xb102e308u  /* RN32(ln 2 - head)                  */
static const uint32_t orc_inv_fact[8] = {
    0x3f800000u, /* 1/0! */
    0x3f800000u, /* 1/1! */
    0x3f000000u, /* 1/2! */
    0x3e2aaaabu, /* RN32(1/3!) */
    0x3d2aaaabu, /* RN32(1/4!) */
    0x3c088889u, /* RN32(1/5!) */
    0x3ab60b61u, /* RN32(1/6!) */
    0x39500d01u, /* RN32(1/7!) */
};

static float pow2i(int n) { /* exact 2^n for n in [-126, 127] */
    return bits_to_f32((uint32_t)(n + 127) << 23);
}

float orc_expf(float x) {
    if (x != x) return x;
    if (x > bits_to_f32(ORC_EXP_HI)) return INFINITY;
    if (x < bits_to_f32(ORC_EXP_LO)) return 0.0f;
    float t = x * bits_to_f32(ORC_LOG2E);
    float n = rintf(t); /* ties to even in the default rounding mode */
    float r = fmaf(-n, bits_to_f32(ORC_LN2_HEAD), x);
    r = fmaf(-n, bits_to_f32(ORC_LN2_TAIL), r);
    float p = bits_to_f32(orc_inv_fact[7]);
    for (int j = 6; j >= 0; --j) p = fmaf(p, r, bits_to_f32(orc_inv_fact[j]));
    int ni = (int)n;
    if (ni > 127) {
        p = p * 2.0f;
        ni -= 1;
    }
    if (ni >= -126) return p * pow2i(ni);
    return (p * pow2i(ni + 64)) * pow2i(-64);
}

void orc_expf_n(const float *x, size_t n, float *out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_expf(x[i]);
}

/* SiLU(gate) * up with silu(g) = g / (1 + e^-g), each step one binary32
 * operation: e = exp(-g); d = 1 + e; s = g / d; act = s * up. */
float orc_silu_mul(float gate, float up) {
    float e = orc_expf(-gate);
    float d = 1.0f + e;
    float s = gate / d;
    return s * up;
}

void orc_silu_mul_n(const float *g, const float *u, size_t n, float *out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_silu_mul(g[i], u[i]);
}

/* ---------------------------------------------------------------------
 * Activation quantisation (w8a8_decode.rs: w8a8_act_quant,
 * w8a8_act_quant_silu, W8a8Scale::act_scales_per_row).  One scale per
 * token row (PerRow) or per 128-wide K group (Block128):
 *   s = absmax / 448          (binary32 division)
 *   q = e4m3(x / s)           (binary32 division, then RNE satfinite)
 * A group whose absmax is 0 stores s = 0 and the codes of its +-0 inputs.
 * ------------------------------------------------------------------- */

static void quant_group(const float *a, int len, uint8_t *q, float *s) {
    float amax = 0.0f;
    for (int i = 0; i < len; ++i) {
        float v = fabsf(a[i]);
        if (v > amax) amax = v;
    }
    float scale = amax / 448.0f;
    *s = scale;
    for (int i = 0; i < len; ++i)
        q[i] = (scale == 0.0f) ? orc_e4m3_encode(a[i])
                               : orc_e4m3_encode(a[i] / scale);
}

static void quant_rows(int fmt, const float *act, int rows, int k, uint8_t *q,
                       float *s) {
    int group = (fmt == ORC_PER_ROW) ? k : 128;
    int per_row = k / group;
    for (int m = 0; m < rows; ++m)
        for (int g = 0; g < per_row; ++g)
            quant_group(act + (size_t)m * k + (size_t)g * group, group,
                        q + (size_t)m * k + (size_t)g * group,
                        s + (size_t)m * per_row + g);
}

void orc_act_quant(int fmt, const uint16_t *x, size_t ldx, int rows, int k,
                   uint8_t *q, float *s) {
    float *act = (float *)malloc_or_die((size_t)rows * k * sizeof(float));
    for (int m = 0; m < rows; ++m)
        for (int i = 0; i < k; ++i)
            act[(size_t)m * k + i] = bf16_to_f32(x[(size_t)m * ldx + i]);
    quant_rows(fmt, act, rows, k, q, s);
    free(act);
}

void orc_act_quant_silu(int fmt, const uint16_t *gate, size_t ld_gate,
                        const uint16_t *up, size_t ld_up, int rows, int k,
                        uint8_t *q, float *s) {
    float *act = (float *)malloc_or_die((size_t)rows * k * sizeof(float));
    for (int m = 0; m < rows; ++m)
        for (int i = 0; i < k; ++i)
            act[(size_t)m * k + i] =
                orc_silu_mul(bf16_to_f32(gate[(size_t)m * ld_gate + i]),
                             bf16_to_f32(up[(size_t)m * ld_up + i]));
    quant_rows(fmt, act, rows, k, q, s);
    free(act);
}

/* ---------------------------------------------------------------------
 * W8A8 GEMV (w8a8_decode.rs: W8a8Weight::new, W8a8Weight::boundaries,
 * w8a8_gemv).  The weight is 1..3 FP8 segments [n_s, K] (K contiguous)
 * concatenated along the output dimension; output column j belongs to
 * segment 0 for j < n1, to segment 1 (row j - n1) for n1 <= j < n2, and to
 * segment 2 (row j - n2) otherwise.
 *   x_hat[m,k] = dec(q[m,k]) * sa(m, k)
 *   w_hat[j,k] = dec(W_s[r,k]) * sw_s(r, k)
 *   y[m,j]     = sum_k x_hat[m,k] * w_hat[j,k]          (double)
 * with sa(m,k) = sa[m] (PerRow) or sa[m, k/128] (Block128), and
 * sw_s(r,k) = sw_s[r] (PerRow) or sw_s[r/128, k/128] (Block128; the
 * segment's scale grid is [ceil(n_s/128), K/128], row-major).
 * bound[m,j] = sum_k |x_hat * w_hat|, the scale of the parity tolerance.
 * ------------------------------------------------------------------- */

/* split points (n1, n2) of the concatenated output, as
 * W8a8Weight::boundaries gives them: one segment (N, N), two (n0, N),
 * three (n0, n0 + n1). */
static void route(int count, const int *n, int j, int *seg, int *row) {
    int N = 0;
    for (int s = 0; s < count; ++s) N += n[s];
    int n1 = (count == 1) ? N : n[0];
    int n2 = (count == 3) ? n[0] + n[1] : N;
    if (j < n1) {
        *seg = 0;
        *row = j;
    } else if (j < n2) {
        *seg = 1;
        *row = j - n1;
    } else {
        *seg = 2;
        *row = j - n2;
    }
}

static void gemv_one(int fmt, const uint8_t *q, const float *sa, int k,
                     int count, const uint8_t *const *w,
                     const float *const *sw, const int *n, int m, int j,
                     double *y, double *bound) {
    int seg, r;
    route(count, n, j, &seg, &r);
    int kb_per_row = k / 128;
    const uint8_t *wrow = w[seg] + (size_t)r * k;
    double acc = 0.0, abs_acc = 0.0;
    for (int kk = 0; kk < k; ++kk) {
        double a_scale = (fmt == ORC_PER_ROW)
                             ? (double)sa[m]
                             : (double)sa[(size_t)m * kb_per_row + kk / 128];
        double w_scale =
            (fmt == ORC_PER_ROW)
                ? (double)sw[seg][r]
                : (double)sw[seg][(size_t)(r / 128) * kb_per_row + kk / 128];
        double xh = (double)orc_e4m3_decode(q[(size_t)m * k + kk]) * a_scale;
        double wh = (double)orc_e4m3_decode(wrow[kk]) * w_scale;
        acc += xh * wh;
        abs_acc += fabs(xh * wh);
    }
    *y = acc;
    *bound = abs_acc;
}

void orc_w8a8_gemv(int fmt, const uint8_t *q, const float *sa, int rows,
                   int k, int count, const uint8_t *const *w,
                   const float *const *sw, const int *n, double *y,
                   double *bound) {
    int N = 0;
    for (int s = 0; s < count; ++s) N += n[s];
#pragma omp parallel for schedule(dynamic, 16)
    for (int j = 0; j < N; ++j)
        for (int m = 0; m < rows; ++m)
            gemv_one(fmt, q, sa, k, count, w, sw, n, m, j,
                     &y[(size_t)m * N + j], &bound[(size_t)m * N + j]);
}

void orc_w8a8_gemv_sampled(int fmt, const uint8_t *q, const float *sa,
                           int rows, int k, int count, const uint8_t *const *w,
                           const float *const *sw, const int *n,
                           const int *sample_row, const int *sample_col,
                           int n_samples, double *y, double *bound) {
    (void)rows;
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < n_samples; ++i)
        gemv_one(fmt, q, sa, k, count, w, sw, n, sample_row[i], sample_col[i],
                 &y[i], &bound[i]);
}

/* ---------------------------------------------------------------------
 * AWQ INT4 fused QKV (fused_int4_qkv.rs).  For each projection p with
 * width n (nq for q, nkv for k and v), column c, reduction index k:
 *   packed = qw[k * (n/8) + c/8]
 *   nib    = (packed >> SHIFT[c % 8]) & 0xF, SHIFT = {0,16,4,20,8,24,12,28}
 *   w      = (f32(nib) - zr[(k/group) * n + c]) * sc[(k/group) * n + c]  (f32)
 *   out[m, c] = sum_k x[m, k] * w                                   (double)
 * ------------------------------------------------------------------- */

static const int orc_awq_shift[8] = {0, 16, 4, 20, 8, 24, 12, 28};

void orc_int4_qkv(const float *x, int m, int k, int nq, int nkv, int group,
                  const uint32_t *const *qw, const float *const *sc,
                  const float *const *zr, double *const *out,
                  double *const *bound) {
    for (int p = 0; p < 3; ++p) {
        int n = (p == 0) ? nq : nkv;
        int n_packed = n / 8;
#pragma omp parallel for schedule(dynamic, 16)
        for (int c = 0; c < n; ++c) {
            for (int row = 0; row < m; ++row) {
                double acc = 0.0, abs_acc = 0.0;
                for (int kk = 0; kk < k; ++kk) {
                    uint32_t packed = qw[p][(size_t)kk * n_packed + c / 8];
                    uint32_t nib = (packed >> orc_awq_shift[c % 8]) & 0xFu;
                    size_t gi = (size_t)(kk / group) * n + c;
                    float wv = ((float)nib - zr[p][gi]) * sc[p][gi];
                    double t = (double)x[(size_t)row * k + kk] * (double)wv;
                    acc += t;
                    abs_acc += fabs(t);
                }
                out[p][(size_t)row * n + c] = acc;
                bound[p][(size_t)row * n + c] = abs_acc;
            }
        }
    }
}

/* ---------------------------------------------------------------------
 * FP8 weight quantisation: the weight side of w8a8_decode.rs's scale
 * layouts (enum W8a8Scale: one f32 scale per output row, or one per 128x128
 * block of the [n, K] weight stored [ceil(n/128), K/128]), with the scale
 * the workloads state for weights, absmax / 448:
 *   s    = absmax over the row or block / 448      (binary32 division)
 *   code = e4m3(w / s)                             (binary32 division, RNE satfinite)
 * A row or block whose absmax is 0 stores s = 0 and the codes of its +-0
 * values (the rule the activation quantiser follows).  A ragged last block
 * row covers the remaining n % 128 rows.
 * ------------------------------------------------------------------- */

static void quant_region(const float *w, size_t ldw, int r0, int r1, int c0, int c1, uint8_t *codes, int k,
                         float *s_out) {
    float amax = 0.0f;
    for (int r = r0; r < r1; ++r)
        for (int c = c0; c < c1; ++c) {
            float v = fabsf(w[(size_t)r * ldw + c]);
            if (v > amax) amax = v;
        }
    float scale = amax / 448.0f;
    *s_out = scale;
    for (int r = r0; r < r1; ++r)
        for (int c = c0; c < c1; ++c) {
            float v = w[(size_t)r * ldw + c];
            codes[(size_t)r * k + c] = (scale == 0.0f) ? orc_e4m3_encode(v) : orc_e4m3_encode(v / scale);
        }
}

void orc_fp8_weight_quant(int fmt, const float *w, size_t ldw, int n, int k, uint8_t *codes, float *scales) {
    if (fmt == ORC_PER_ROW) {
#pragma omp parallel for schedule(static)
        for (int r = 0; r < n; ++r) quant_region(w, ldw, r, r + 1, 0, k, codes, k, scales + r);
    } else {
        int nb = (n + 127) / 128, kb = k / 128;
#pragma omp parallel for schedule(static)
        for (int b = 0; b < nb * kb; ++b) {
            int br = b / kb, bc = b % kb;
            int r1 = (br + 1) * 128 < n ? (br + 1) * 128 : n;
            quant_region(w, ldw, br * 128, r1, bc * 128, bc * 128 + 128, codes, k, scales + b);
        }
    }
}

/* AWQ packing, the inverse of the unpacking in fused_int4_qkv.rs
 * (QKV_AWQ_SHIFTS, unpack_awq_qkv): word j of row kk holds the code of
 * column 8j + i at bits SHIFT[i] .. SHIFT[i] + 3.  Codes are 0..15, one per
 * byte of nib [k, n]; qw is [k, n/8]. */
void orc_awq_pack(const uint8_t *nib, int k, int n, uint32_t *qw) {
    int words = n / 8;
    for (int kk = 0; kk < k; ++kk)
        for (int j = 0; j < words; ++j) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i)
                word |= (uint32_t)(nib[(size_t)kk * n + 8 * j + i] & 0xFu) << orc_awq_shift[i];
            qw[(size_t)kk * words + j] = word;
        }
}

/* ---------------------------------------------------------------------
 * KV-cache quantisation (kv_cache_quant.wgsl).
 *
 * Per-token symmetric int8 (the page's quantize_kv_fp8_per_token_f32 and
 * quantize_kv_int8_f32 compute the same thing; the "FP8" name does not match
 * its arithmetic, which scales to 127 and rounds to integers): per token row,
 *   s = max(absmax / 127, 1e-8),  q = clamp(round(v / s), -128, 127)
 * with WGSL round() (nearest integer, halves to even); dequantisation is
 * q * s.  The page stores each code in its own u32 word; here codes are int8
 * bytes, the same values.
 *
 * Per-group asymmetric INT4 (quantize_kv_int4_f32 / dequantize_kv_int4_f32):
 * groups are consecutive runs of `group` values of the flattened
 * [tokens, head_dim] array;
 *   scale = (max - min) / 15,  zero = -min / max(scale, 1e-8),
 *   q = clamp(round((v - min) / max(scale, 1e-8)), 0, 15),
 *   dequantised v = q * scale - zero * scale.
 * Two codes per byte: flattened element e sits in byte e / 2, the low nibble
 * for even e.  The page writes zeros at scales[num_tokens + group], which
 * overlaps the scales once there are more groups than tokens; here zeros
 * have an array of their own.
 *
 * Every step is one binary32 operation rounded to nearest (the file is
 * built without contraction), so codes and dequantised values are exact.
 * ------------------------------------------------------------------- */

/* WGSL round(): nearest integer, halves to even, for any finite float */
static double round_wgsl(float v) {
    double a = fabs((double)v);
    double r = round_half_even(a);
    return v < 0 ? -r : r;
}

void orc_kv_quant_int8(const float *x, int tokens, int dim, int8_t *q, float *s) {
    for (int t = 0; t < tokens; ++t) {
        const float *row = x + (size_t)t * dim;
        float mx = 0.0f;
        for (int d = 0; d < dim; ++d) {
            float a = fabsf(row[d]);
            if (a > mx) mx = a;
        }
        float sc = mx / 127.0f;
        if (!(sc > 1e-8f)) sc = 1e-8f;
        s[t] = sc;
        for (int d = 0; d < dim; ++d) {
            float r = row[d] / sc;
            double qi = round_wgsl(r);
            if (qi < -128.0) qi = -128.0;
            if (qi > 127.0) qi = 127.0;
            q[(size_t)t * dim + d] = (int8_t)qi;
        }
    }
}

void orc_kv_dequant_int8(const int8_t *q, const float *s, int tokens, int dim, float *out) {
    for (int t = 0; t < tokens; ++t)
        for (int d = 0; d < dim; ++d) {
            size_t i = (size_t)t * dim + d;
            out[i] = (float)q[i] * s[t];
        }
}

void orc_kv_quant_int4(const float *x, size_t n, int group, uint8_t *packed, float *scale, float *zero) {
    size_t groups = n / (size_t)group;
    memset(packed, 0, n / 2);
    for (size_t g = 0; g < groups; ++g) {
        const float *v = x + g * (size_t)group;
        float mn = v[0], mx = v[0];
        for (int i = 0; i < group; ++i) {
            if (v[i] < mn) mn = v[i];
            if (v[i] > mx) mx = v[i];
        }
        float sc = (mx - mn) / 15.0f;
        float den = sc > 1e-8f ? sc : 1e-8f;
        float z = -mn / den;
        scale[g] = sc;
        zero[g] = z;
        for (int i = 0; i < group; ++i) {
            float r = (v[i] - mn) / den;
            double qi = round_wgsl(r);
            if (qi < 0.0) qi = 0.0;
            if (qi > 15.0) qi = 15.0;
            size_t e = g * (size_t)group + (size_t)i;
            if (e % 2 == 0)
                packed[e / 2] = (uint8_t)((packed[e / 2] & 0xF0) | (uint8_t)qi);
            else
                packed[e / 2] = (uint8_t)((packed[e / 2] & 0x0F) | ((uint8_t)qi << 4));
        }
    }
}

void orc_kv_dequant_int4(const uint8_t *packed, const float *scale, const float *zero, size_t n, int group,
                         float *out) {
    for (size_t e = 0; e < n; ++e) {
        size_t g = e / (size_t)group;
        uint8_t b = packed[e / 2];
        int qi = (e % 2) ? (b >> 4) & 0xF : b & 0xF;
        float a = (float)qi * scale[g];
        float c = zero[g] * scale[g];
        out[e] = a - c;
    }
}
