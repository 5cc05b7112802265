/*
 * qdl oracle: plain, slow CPU reference of the quantized decode-time linear
 * layer.  TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What each function follows:
 *   - FP8 E4M3 ("fn" variant: bias 7, max finite 448, no infinities, NaN =
 *     S.1111.111) from the OCP 8-bit floating point specification, rounded
 *     to nearest, ties to even, saturating to +-448 (the reading fixed for
 *     this library because the pages leave the conversion open).
 *   - Activation quantisation per token row or per 128-wide K group, scale
 *     = absmax / 448, from w8a8_decode.rs (W8a8Scale::act_scales_per_row,
 *     w8a8_act_quant).
 *   - SiLU(gate) * up fused before quantisation, from w8a8_decode.rs
 *     (w8a8_act_quant_silu); the exponential is the library's own written
 *     specification (qdl exp, below), so the codes are reproducible.
 *   - The W8A8 GEMV over 1..3 row-concatenated FP8 weight segments with
 *     per-row or 128x128 block scales, from w8a8_decode.rs (W8a8Weight::new,
 *     W8a8Weight::boundaries, w8a8_gemv), as dequantise-then-dot in double.
 *   - The AWQ INT4 fused-QKV GEMV of fused_int4_qkv.rs (QKV_AWQ_SHIFTS,
 *     unpack_awq_qkv, fused_int4_qkv_q/_k/_v): f32 dequantisation exactly as
 *     the shader writes it, dot product accumulated in double.
 *   - FP8 weight quantisation per output row or 128x128 block with scale
 *     absmax / 448 (the weight recipe of the workloads, in the scale layouts
 *     of w8a8_decode.rs), and AWQ packing of 4-bit codes in the shift order
 *     of fused_int4_qkv.rs (the inverse of its unpacking).
 *   - The KV-cache quantisers of kv_cache_quant.wgsl: per-token symmetric
 *     int8 and per-group asymmetric INT4 with two codes per byte, and their
 *     dequantisers, step for step in binary32.
 *
 * Parity pins: every function is checked against values fixed by the pages
 * and the mathematics in tests/test_oracle_*.py (hand-computed nibble and
 * FP8 cases, a library FP8 conversion, brute force over the FP8 grid,
 * double-precision exp, special cases reducing to a library matmul).
 */
#ifndef QDL_ORACLE_H
#define QDL_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* weight/activation scale layouts (w8a8_decode.rs, enum W8a8Scale) */
#define ORC_PER_ROW 0
#define ORC_BLOCK128 1

uint8_t orc_e4m3_encode(float v);
float orc_e4m3_decode(uint8_t code);
void orc_e4m3_encode_n(const float *v, size_t n, uint8_t *out);
void orc_e4m3_decode_n(const uint8_t *c, size_t n, float *out);

float orc_expf(float x);
void orc_expf_n(const float *x, size_t n, float *out);
float orc_silu_mul(float gate, float up);
void orc_silu_mul_n(const float *g, const float *u, size_t n, float *out);

/* x: bf16 bit patterns [rows, ldx]; q: [rows, k]; s: [rows] (PER_ROW) or
 * [rows, k/128] (BLOCK128). */
void orc_act_quant(int fmt, const uint16_t *x, size_t ldx, int rows, int k,
                   uint8_t *q, float *s);
void orc_act_quant_silu(int fmt, const uint16_t *gate, size_t ld_gate,
                        const uint16_t *up, size_t ld_up, int rows, int k,
                        uint8_t *q, float *s);

/* y, bound: [rows, N] with N = sum of n[]; bound = sum_k |x_hat * w_hat|. */
void orc_w8a8_gemv(int fmt, const uint8_t *q, const float *sa, int rows,
                   int k, int count, const uint8_t *const *w,
                   const float *const *sw, const int *n, double *y,
                   double *bound);

/* y[j] for a list of (row, output column) samples only. */
void orc_w8a8_gemv_sampled(int fmt, const uint8_t *q, const float *sa,
                           int rows, int k, int count, const uint8_t *const *w,
                           const float *const *sw, const int *n,
                           const int *sample_row, const int *sample_col,
                           int n_samples, double *y, double *bound);

/* x: f32 [m, k]; qw[p]: u32 [k, n_p/8]; sc[p], zr[p]: f32 [k/group, n_p];
 * out[p], bound[p]: [m, n_p], with n_0 = nq, n_1 = n_2 = nkv. */
void orc_int4_qkv(const float *x, int m, int k, int nq, int nkv, int group,
                  const uint32_t *const *qw, const float *const *sc,
                  const float *const *zr, double *const *out,
                  double *const *bound);

/* FP8 weight quantisation per output row or per 128x128 block (scale =
 * absmax / 448): w f32 [n, ldw] (first k columns), k % 128 == 0;
 * codes [n, k]; scales [n] (PER_ROW) or [ceil(n/128), k/128] (BLOCK128). */
void orc_fp8_weight_quant(int fmt, const float *w, size_t ldw, int n, int k, uint8_t *codes, float *scales);

/* AWQ packing in the shift order of fused_int4_qkv.rs: nib u8 [k, n] (codes
 * 0..15, n % 8 == 0) -> qw u32 [k, n/8]. */
void orc_awq_pack(const uint8_t *nib, int k, int n, uint32_t *qw);

/* KV-cache quantisation (kv_cache_quant.wgsl): per-token symmetric int8,
 * x [tokens, dim] -> q int8 [tokens, dim], s [tokens]; per-group asymmetric
 * INT4 over the flattened x [n] (n % group == 0, group even) -> packed
 * [n / 2] (two codes per byte, even element in the low nibble), scale and
 * zero [n / group]. */
void orc_kv_quant_int8(const float *x, int tokens, int dim, int8_t *q, float *s);
void orc_kv_dequant_int8(const int8_t *q, const float *s, int tokens, int dim, float *out);
void orc_kv_quant_int4(const float *x, size_t n, int group, uint8_t *packed, float *scale, float *zero);
void orc_kv_dequant_int4(const uint8_t *packed, const float *scale, const float *zero, size_t n, int group,
                         float *out);

int orc_num_threads(void);
/* threads for later parallel loops (OpenMP); no effect in a serial build */
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
