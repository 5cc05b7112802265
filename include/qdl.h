/*
 * libqdl -- quantized decode-time linear layer for NVIDIA GB300 (sm_103a).
 *
 * Two variants of the decode-time projection y = x W^T:
 *
 *   W8A8   FP8 E4M3 activations (quantised here, per token row or per
 *          128-wide K group, optionally with SiLU(gate)*up fused in) times an
 *          FP8 E4M3 weight with per-row or 128x128-block f32 scales, made of
 *          1..3 segments concatenated along the output dimension.
 *          Defined by w8a8_decode.rs (metrale_model_layers, layers::ops).
 *   W4A16  AWQ INT4 fused Q/K/V projection with per-group scales and zeros.
 *          Defined by fused_int4_qkv.rs (boostr, quant::wgpu::shaders).
 *
 * Weights are read-only inputs: the decode entry points start streaming
 * weight codes (and AWQ codes, scales and zeros) as soon as they launch,
 * before they wait for the kernel ahead of them on the stream, so weights
 * must be written by work that has finished by then -- anything that does
 * not release its dependents early, such as qdl_fp8_weight_quant,
 * qdl_awq_pack, a copy or an ordinary kernel.  Activations, scratch and
 * outputs are touched only after that wait.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are device pointers owned by the caller; the
 *     library never allocates, frees or retains them.  Layouts are row-major
 *     with the strides given.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronises.
 *   - Every call validates all arguments on the host before it touches the
 *     device.  On any error nothing is launched, the call returns a non-zero
 *     qdl_status and qdl_last_error() returns a message for the calling
 *     thread.  Kernel launch failures return QDL_ERR_CUDA.
 *   - FP8 E4M3 is the OCP "E4M3" format (bias 7, max finite 448, no inf,
 *     NaN = S.1111.111).  Activation codes are produced by
 *     round-to-nearest-even with saturation to +-448.
 */
#ifndef QDL_H
#define QDL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QDL_API __attribute__((visibility("default")))
#else
#define QDL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QDL_OK = 0,
    QDL_ERR_INVALID_ARG = 1,       /* a shape, stride, pointer or enum is invalid */
    QDL_ERR_SCRATCH_TOO_SMALL = 2, /* activation buffers cannot hold rows x K   */
    QDL_ERR_UNSUPPORTED = 3,       /* valid per the definition, beyond a limit  */
    QDL_ERR_CUDA = 4,              /* the CUDA runtime reported an error        */
    QDL_ERR_DEVICE_TIMEOUT = 5     /* a bounded device-side wait gave up        */
} qdl_status;

/* Scale layouts, w8a8_decode.rs enum W8a8Scale.
 *   PER_ROW : one f32 weight scale per output row; one activation scale per
 *             token row.
 *   BLOCK128: one f32 weight scale per 128x128 block of each segment, stored
 *             [ceil(n_s/128), K/128] row-major; one activation scale per
 *             token row and 128-wide K group, stored [rows, K/128]. */
typedef enum { QDL_SCALE_PER_ROW = 0, QDL_SCALE_BLOCK128 = 1 } qdl_scale;

/* Output element type of the W8A8 GEMV.  QDL_OUT_F32_ADD (qdl_w8a8_gemv
 * only) adds y to the f32 values already in out; split-K partial sums are
 * then added with f32 atomics, so their order, and the last bits of the
 * result, may vary from run to run.  QDL_OUT_F32_DETERMINISTIC writes f32
 * like QDL_OUT_F32, but the projections then never add split-K partials
 * with atomics: they meet in a fixed-order reduction, so identical calls
 * give identical bits (for callers that compare logits across runs), at the
 * cost of the cluster reduction's time where K is split. */
typedef enum {
    QDL_OUT_F32 = 0,
    QDL_OUT_BF16 = 1,
    QDL_OUT_F32_ADD = 2,
    QDL_OUT_F32_DETERMINISTIC = 3
} qdl_dtype;

#define QDL_MAX_ROWS 256  /* w8a8_decode.rs W8A8_MAX_ROWS */
#define QDL_K_UNIT 128    /* w8a8_decode.rs W8A8_K_UNIT   */
#define QDL_MAX_K 65536   /* library limit on K for the activation quantiser */
#define QDL_MAX_PROJ_ROWS 65536 /* library limit on rows of one qdl_w8a8_proj call */

/* One FP8 weight segment (the fields w8a8_decode.rs reads from Fp8Weight).
 *   weight : device, e4m3 codes [n, k], row-major (K contiguous), 16-byte
 *            aligned.
 *   scale  : device, f32, [n] (PER_ROW) or [ceil(n/128), k/128] (BLOCK128).
 *   format : qdl_scale of this segment; all segments must agree. */
typedef struct {
    const uint8_t *weight;
    const float *scale;
    uint32_t n;
    uint32_t k;
    int32_t format;
} qdl_fp8_segment;

/* A validated W8A8 weight: 1..3 segments concatenated along N (w8a8_decode.rs
 * struct W8a8Weight).  Fill only through qdl_w8a8_weight_init. */
typedef struct {
    qdl_fp8_segment segs[3];
    uint32_t count;
    uint32_t n;  /* total output width, sum of segment n */
    uint32_t k;
    int32_t format;
    uint32_t n1, n2; /* split points, W8a8Weight::boundaries */
    uint32_t magic;  /* set by qdl_w8a8_weight_init */
} qdl_w8a8_weight;

/* W8a8Weight::new.  Checks: 1 <= count <= 3; every segment has the same k
 * and format; k > 0 and k % 128 == 0; format is PER_ROW or BLOCK128; every
 * n > 0 with non-NULL weight and scale; every segment but the last has n a
 * multiple of 16 (PER_ROW) or 128 (BLOCK128) (W8a8Scale::segment_align);
 * weight pointers 16-byte aligned and scale pointers 4-byte aligned; the
 * total n fits in 2^31.  Output column j maps to segment 0 for j < n1, to
 * segment 1 (row j - n1) for n1 <= j < n2, to segment 2 (row j - n2) after;
 * (n1, n2) = (N, N), (n0, N) or (n0, n0 + n1) for 1, 2 or 3 segments.
 * Reads host memory only. */
QDL_API qdl_status qdl_w8a8_weight_init(qdl_w8a8_weight *out, const qdl_fp8_segment *segs,
                                uint32_t count);

/* Activation buffer sizes for up to QDL_MAX_ROWS rows of K <= max_k
 * (W8a8Scratch::alloc): q_bytes = 256 * max_k, scale_bytes =
 * 256 * max(ceil(max_k / 128), 1) * 4.  Either output pointer may be NULL. */
QDL_API qdl_status qdl_scratch_bytes(uint32_t max_k, size_t *q_bytes, size_t *scale_bytes);

/* Activation quantisation (w8a8_decode.rs fn w8a8_act_quant).
 *   x       : device bf16 [rows, ldx]; columns 0..k-1 of each row are read.
 *   q       : device e4m3 codes [rows, k] (row stride k), q_bytes capacity.
 *   q_scale : device f32 [rows] (PER_ROW) or [rows, k/128] (BLOCK128),
 *             scale_bytes capacity.
 * s = absmax / 448 (binary32 division); q = e4m3_rne_sat(x / s); a group
 * whose absmax is 0 gets s = 0 and the codes of its signed zeros.
 * Checks: 1 <= rows <= 256; q_bytes >= rows*k and scale_bytes >= rows *
 * scales_per_row * 4 (else QDL_ERR_SCRATCH_TOO_SMALL); k % 128 == 0,
 * k <= QDL_MAX_K, ldx >= k, ldx % 8 == 0, x 16-byte aligned, q 16-byte
 * aligned, q_scale 4-byte aligned. */
QDL_API qdl_status qdl_act_quant(int32_t format, const void *x, uint32_t ldx, uint32_t rows,
                         uint32_t k, uint8_t *q, float *q_scale, size_t q_bytes,
                         size_t scale_bytes, void *stream);

/* Activation quantisation of act = SiLU(gate) * up (w8a8_decode.rs fn
 * w8a8_act_quant_silu), silu(g) = g / (1 + e^-g).  Each step is one binary32
 * operation (e = exp(-g), d = 1 + e, s = g / d, act = s * up) with the
 * library's own exp (Cody and Waite reduction, degree-7 Taylor polynomial;
 * specified in the source), so the codes are reproducible bit for bit.
 * gate, up: device bf16 [rows, ld_gate] / [rows, ld_up]; they may be two
 * column ranges of one buffer.  Same checks as qdl_act_quant, per stride. */
QDL_API qdl_status qdl_act_quant_silu(int32_t format, const void *gate, const void *up,
                              uint32_t ld_gate, uint32_t ld_up, uint32_t rows, uint32_t k,
                              uint8_t *q, float *q_scale, size_t q_bytes, size_t scale_bytes,
                              void *stream);

/* W8A8 GEMV / skinny GEMM (w8a8_decode.rs fn w8a8_gemv):
 *   y[m, j] = sum_k dec(q[m,k]) sa(m,k) dec(W[j,k]) sw(j,k)
 * with the scale layouts of qdl_scale, over all rows (one pass over the
 * weights for any rows <= 256).
 *   q, q_scale : device, as written by qdl_act_quant (capacities q_bytes,
 *                scale_bytes are checked like the activation scratch).
 *   out        : device [rows, ldc] of out_dtype (f32, or bf16 rounded to
 *                nearest even, or f32 accumulated: out += y); columns
 *                N..ldc-1 are not written.
 * With F32 and BF16 output, the partial sums of CTAs that split K are added
 * in a fixed order, so results are reproducible bit for bit.
 * Checks: weight initialised; 1 <= rows <= 256; capacities; ldc >= N;
 * out aligned to its element size; out_dtype valid. */
QDL_API qdl_status qdl_w8a8_gemv(const qdl_w8a8_weight *w, const uint8_t *q, const float *q_scale,
                         size_t q_bytes, size_t scale_bytes, uint32_t rows, void *out,
                         int32_t out_dtype, uint32_t ldc, void *stream);

/* Decode projection (w8a8_decode.rs fn w8a8_proj): qdl_act_quant with the
 * weight's format and K, then qdl_w8a8_gemv, on one stream.  q and q_scale
 * are the caller's activation scratch (sizes from qdl_scratch_bytes).
 * rows may exceed 256 (a prefill-shaped call; the page stops at
 * W8A8_MAX_ROWS = 256), up to QDL_MAX_PROJ_ROWS.  When q_bytes and
 * scale_bytes hold all rows (rows * k and rows * scales_per_row * 4 bytes),
 * the rows are quantised into them 256 at a time and one GEMV launch covers
 * every row, streaming the weights once.  Otherwise the call runs in passes
 * of 256 rows, in order on the stream, each quantising into the same 256-row
 * scratch and streaming the weights once more; pass p covers rows 256p.. of
 * x and out.  The scratch needs to hold min(rows, 256) rows.
 * With f32 output, when the GEMV splits K over several CTAs, the quantiser
 * first sets out[0..rows)[0..N) to zero and the GEMV adds into it
 * (QDL_OUT_F32_ADD): the order of the split-K additions varies, so results
 * may differ in the last bits from run to run (always within the GEMV's
 * error bound).  bf16 output and QDL_OUT_F32_DETERMINISTIC take the
 * fixed-order reduction and are reproducible bit for bit.  out_dtype is
 * QDL_OUT_F32, QDL_OUT_BF16 or QDL_OUT_F32_DETERMINISTIC.  Checks: those of
 * qdl_w8a8_gemv, plus the
 * quantiser's K <= QDL_MAX_K and the x checks of qdl_act_quant. */
QDL_API qdl_status qdl_w8a8_proj(const qdl_w8a8_weight *w, const void *x, uint32_t ldx, uint32_t rows,
                         void *out, int32_t out_dtype, uint32_t ldc, uint8_t *q, float *q_scale,
                         size_t q_bytes, size_t scale_bytes, void *stream);

/* MLP down projection: qdl_act_quant_silu with the weight's format and K,
 * then qdl_w8a8_gemv (the composition w8a8_decode.rs uses for gate/up
 * inputs).  f32 output is accumulated, and rows beyond 256 run in passes,
 * as in qdl_w8a8_proj. */
QDL_API qdl_status qdl_w8a8_proj_silu(const qdl_w8a8_weight *w, const void *gate, const void *up,
                              uint32_t ld_gate, uint32_t ld_up, uint32_t rows, void *out,
                              int32_t out_dtype, uint32_t ldc, uint8_t *q, float *q_scale,
                              size_t q_bytes, size_t scale_bytes, void *stream);

/* AWQ INT4 fused Q/K/V projection (fused_int4_qkv.rs: fused_int4_qkv_q,
 * fused_int4_qkv_k, fused_int4_qkv_v, unpack_awq_qkv).  For projection p
 * (0 = q with width nq, 1 = k and 2 = v with width nkv), column c, row i:
 *   nib = (qw[p][kk * (n/8) + c/8] >> SHIFT[c % 8]) & 0xF,
 *         SHIFT = {0, 16, 4, 20, 8, 24, 12, 28}
 *   w   = (nib - zr[p][(kk/group) * n + c]) * sc[p][(kk/group) * n + c]
 *   out[p][i * n + c] = sum_kk x[i * k + kk] * w
 *   x      : device f32 [m, k], 16-byte aligned, |x| < 65504.
 *   qw[p]  : device u32 [k, n/8], 4-byte aligned (8-byte aligned with
 *            nq, nkv multiples of 16 enables 8-byte weight loads).
 *   sc[p], zr[p] : device f32 [k/group, n], 16-byte aligned.
 *   out[p] : device f32 [m, n], 4-byte aligned.
 * With nq and nkv multiples of 32 and every qw[p] 16-byte aligned, up to 4
 * rows (up to 8 with group != 128) take one CUDA-core pass in f32 (x
 * unrounded, exact nibbles), and more rows with group 128 take the tcgen05
 * kernel once per 16 rows, which
 * multiplies x rounded to f16 with exact nibbles (error within 2^-11 of
 * sum |x w|) and applies zeros and scales per group in f32.  Both make two
 * launches: out is zeroed, then the GEMV adds per-tile partial sums into it
 * with f32 atomics, so the order of those additions, and the last bits of
 * the result, vary from run to run.  Every other shape takes an mma.sync
 * kernel (x rounded to f16) once per 16 rows.
 * Checks: m >= 1; k >= 1; group > 0,
 * group % 16 == 0, k % group == 0; nq, nkv > 0 and multiples of 8; no NULL
 * pointer; alignments above. */
QDL_API qdl_status qdl_int4_qkv_gemv(const float *x, uint32_t m, uint32_t k, uint32_t nq, uint32_t nkv,
                             uint32_t group, const uint32_t *const *qw, const float *const *sc,
                             const float *const *zr, float *const *out, void *stream);

/* ------------------------------------------------------------------
 * KV-cache quantisers (kv_cache_quant.wgsl: quantize_kv_fp8_per_token_f32,
 * quantize_kv_int8_f32, quantize_kv_int4_f32 and the dequantize_* kernels).
 * The page's "FP8" per-token kernel and its INT8 one compute the same thing,
 * symmetric int8, so one pair of entry points serves both.  Every step is
 * one binary32 operation rounded to nearest; round() takes halves to even.
 * Arguments are device pointers; calls are asynchronous on `stream`; on an
 * invalid argument nothing is launched and qdl_last_error() explains.
 * Shapes: x and out are [tokens, head_dim] f32 (row-major, 16-byte aligned);
 * tokens >= 1, head_dim a positive multiple of 4, tokens * head_dim < 2^31.
 * ------------------------------------------------------------------ */

/* Per token t:  scale[t] = max(absmax_d |x[t,d]| / 127, 1e-8),
 *               q[t,d] = clamp(round(x[t,d] / scale[t]), -128, 127).
 * q: int8 [tokens, head_dim] (the page keeps each code in a u32 word; the
 * values are the same), 4-byte aligned; scale: f32 [tokens]. */
QDL_API qdl_status qdl_kv_quant_int8(const float *x, uint32_t tokens, uint32_t head_dim, int8_t *q, float *scale,
                                     void *stream);

/* out[t,d] = q[t,d] * scale[t]. */
QDL_API qdl_status qdl_kv_dequant_int8(const int8_t *q, const float *scale, uint32_t tokens, uint32_t head_dim,
                                       float *out, void *stream);

/* Per group g of `group` consecutive values of the flattened x (group a
 * positive multiple of 8 dividing tokens * head_dim):
 *   scale[g] = (max - min) / 15,  zero[g] = -min / max(scale[g], 1e-8),
 *   code = clamp(round((v - min) / max(scale[g], 1e-8)), 0, 15).
 * packed: [tokens * head_dim / 2] bytes, two codes per byte, value e in byte
 * e / 2, the low nibble when e is even; 4-byte aligned.  scale, zero: f32
 * [tokens * head_dim / group], separate arrays (the page stores zeros after
 * the scales at an offset of num_tokens, which overlaps the scales as soon as
 * there are more groups than tokens).  A constant group gets scale 0 and
 * dequantises to 0, as the page's formulas give. */
QDL_API qdl_status qdl_kv_quant_int4(const float *x, uint32_t tokens, uint32_t head_dim, uint32_t group,
                                     uint8_t *packed, float *scale, float *zero, void *stream);

/* out[e] = code(e) * scale[g] - zero[g] * scale[g], g = e / group. */
QDL_API qdl_status qdl_kv_dequant_int4(const uint8_t *packed, const float *scale, const float *zero, uint32_t tokens,
                                       uint32_t head_dim, uint32_t group, float *out, void *stream);

/* ------------------------------------------------------------------
 * Weight preparation.  The decode path takes FP8 and AWQ weights as inputs;
 * these entry points make them on the GPU.  Arguments are device pointers;
 * calls are asynchronous on `stream`; on an invalid argument nothing is
 * launched and qdl_last_error() explains.
 * ------------------------------------------------------------------ */

/* Element type of a weight to quantise. */
typedef enum { QDL_IN_F32 = 0, QDL_IN_BF16 = 1 } qdl_in_dtype;

/* FP8 E4M3 weight in the scale layouts of w8a8_decode.rs (enum W8a8Scale),
 * with the scale the workloads state for weights:
 *   PER_ROW : s[r] = absmax_k |w[r,k]| / 448, one per output row;
 *   BLOCK128: s[i, j] = absmax over rows 128i.. and columns 128j.. / 448,
 *             stored [ceil(n/128), k/128]; the last block row covers the
 *             remaining n % 128 rows;
 *   code    = e4m3(w / s), both divisions binary32, round to nearest even,
 *             saturating to +-448; a row or block whose absmax is 0 gets
 *             s = 0 and the codes of its signed zeros.
 *   w      : device [n, ldw] of w_dtype (qdl_in_dtype), columns 0..k-1 read;
 *            16-byte aligned, ldw >= k and a multiple of 4 (f32) or 8 (bf16).
 *   codes  : device [n, k] (row stride k), 8-byte aligned.
 *   scales : device f32 [n] or [ceil(n/128), k/128], 4-byte aligned.
 * The result is exactly what qdl_w8a8_weight_init's segments expect.
 * Checks: format and w_dtype valid; n >= 1; k a positive multiple of 128;
 * ldw and alignments above. */
QDL_API qdl_status qdl_fp8_weight_quant(int32_t format, const void *w, int32_t w_dtype, uint32_t ldw, uint32_t n,
                                        uint32_t k, uint8_t *codes, float *scales, void *stream);

/* AWQ packing in the shift order of fused_int4_qkv.rs (QKV_AWQ_SHIFTS, the
 * inverse of unpack_awq_qkv): word j of row kk holds the code of column
 * 8j + i at bits SHIFT[i] .. SHIFT[i] + 3, SHIFT = {0, 16, 4, 20, 8, 24, 12, 28}.
 *   nib : device u8 [k, n], one 4-bit code per byte (only the low 4 bits
 *         are used), 8-byte aligned.
 *   qw  : device u32 [k, n/8], the layout qdl_int4_qkv_gemv reads; 4-byte
 *         aligned.
 * Checks: k >= 1; n a positive multiple of 8; alignments above. */
QDL_API qdl_status qdl_awq_pack(const uint8_t *nib, uint32_t k, uint32_t n, uint32_t *qw, void *stream);

/* Size of the library's own device array used by qdl_w8a8_proj_static. */
#define QDL_STATIC_SCRATCH_BYTES (4 << 20)

/* Decode projection that allocates nothing: qdl_w8a8_proj without caller
 * scratch.  The pages have no counterpart; this entry point exists for
 * callers that cannot allocate device memory -- for example a plugin that a
 * host framework hands only its input and output buffers (the framework owns
 * every allocation and offers no workspace), or a latency-critical decode
 * loop that may not risk cudaMalloc's implicit device synchronisation or an
 * allocation failure mid-step.
 *   The activation codes and scales are kept in one device array built into
 * the library, QDL_STATIC_SCRATCH_BYTES (4 MiB) long, which every GPU that
 * loads the library holds until the process exits.  Calls need
 * rows*K bytes (rounded up to 256) plus rows*scales_per_row*4 bytes of it;
 * larger calls return QDL_ERR_UNSUPPORTED (256 rows fit up to K = 15872).
 *   The first call on a device, made with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  The address is kept for the life of the process, so
 * the library must not be used on a device after cudaDeviceReset there.
 * The call never uses cudaMalloc, cudaFree or any allocating routine.
 *   All calls share the one array and it keeps the last call's contents:
 * calls that can overlap on the GPU (different streams, or several host
 * threads) race on it and must be serialised by the caller.  Each call
 * overwrites every byte it later reads, so no clearing is needed.
 * Arguments and checks are those of qdl_w8a8_proj for w, x, ldx, rows, out,
 * out_dtype and ldc (rows at most 256, K <= QDL_MAX_K). */
QDL_API qdl_status qdl_w8a8_proj_static(const qdl_w8a8_weight *w, const void *x, uint32_t ldx,
                                        uint32_t rows, void *out, int32_t out_dtype, uint32_t ldc,
                                        void *stream);

/* Launch plan of qdl_w8a8_gemv (QDL_OUT_F32) for `rows` token rows on the current device:
 * which kernel runs and how the work is cut (no counterpart on the pages;
 * for tuning and tests).  Queries the device's occupancy tables; launches
 * nothing. */
typedef struct {
    int32_t kernel;      /* 0 = tcgen05 (tensor memory); the only W8A8 kernel */
    uint32_t mma_n;      /* token columns per MMA (tcgen05: 16..256) */
    uint32_t tiles;      /* 128-row output tiles */
    uint32_t split_k;    /* CTAs per tile along K: one cluster, except where the projection's
                            accumulating GEMV (16-token bucket, >= 16 MB of weights) adds
                            the ranks' partials into out and launches them unclustered */
    uint32_t stages;     /* shared-memory pipeline stages per CTA */
    uint32_t threads;    /* threads per CTA */
    uint32_t smem_bytes; /* dynamic shared memory per CTA */
    int32_t resident_clusters; /* clusters of split_k CTAs that fit the device at once */
    uint32_t proj_launches; /* kernels one qdl_w8a8_proj call makes for these rows: the
                               quantiser, then the GEMV (2) */
    uint32_t proj_accumulates; /* 1 when qdl_w8a8_proj with f32 output zeroes out and runs the
                                  GEMV as QDL_OUT_F32_ADD (split K, or the stream-K kernel
                                  that Block128 takes for 17..128 rows), else 0; with its ranks
                                  adding atomically the GEMV may split K where the plain
                                  GEMV's plan (split_k) does not (129..256 rows) */
    uint32_t proj_streamk;     /* 1 when that accumulating GEMV is the stream-K kernel (one
                                  contiguous range of (tile, K block) units per CTA), else 0 */
} qdl_plan;

QDL_API qdl_status qdl_w8a8_plan(const qdl_w8a8_weight *w, uint32_t rows, qdl_plan *plan);

/* Reads and clears the device-side fault word that bounded waits in the
 * kernels set when they give up (synchronises `stream`).  Returns QDL_OK or
 * QDL_ERR_DEVICE_TIMEOUT. */
QDL_API qdl_status qdl_check_device_fault(void *stream);

/* Self-test of the bounded device-side waits (no counterpart on the pages).
 * Runs qdl_w8a8_gemv on valid arguments (ldc = N) with its first pipeline
 * stage deliberately never loaded, so the kernel's waits give up after
 * limit_us microseconds (1..1000000); the kernel records the timeout,
 * drains its in-flight copies with bounded waits and returns normally, and
 * the call then reads the fault word like qdl_check_device_fault.  Returns
 * QDL_ERR_DEVICE_TIMEOUT when the mechanism worked.  `out` receives
 * unspecified values.  Synchronises `stream`. */
QDL_API qdl_status qdl_selftest_bounded_wait(const qdl_w8a8_weight *w, const uint8_t *q,
                                             const float *q_scale, size_t q_bytes,
                                             size_t scale_bytes, uint32_t rows, float *out,
                                             uint32_t limit_us, void *stream);

/* Message for the last error on the calling thread ("" if none). */
QDL_API const char *qdl_last_error(void);

/* Static name of a status code. */
QDL_API const char *qdl_status_string(qdl_status s);

#ifdef __cplusplus
}
#endif
#endif
