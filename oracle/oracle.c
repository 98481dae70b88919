/*
 * oracle.c -- plain, slow, CPU reference for the FP8 W8A8 rollout linear path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU library shares
 * no code, header, table or constant with it, and neither links the other.
 *
 * What it follows (page titles and sections of the FP8-RL pages):
 *  - "FP8-RL: A Practical and Stable Low-Precision Stack for LLM Reinforcement
 *    Learning", section "Prerequisites / FP8 quantisation format": E4M3 with a
 *    range of about [-448, 448]; weights quantised per 128x128 sub-block, one
 *    scale per block, W_hat = round(W / scale).
 *  - same page, "Method steps", step 1: weights are quantised statically at
 *    sync time, activations dynamically in every forward pass; the linears run
 *    as W8A8 (FP8 x FP8) matmuls.
 *  - same page, "Results" (scale-format ablation): fp32 scales versus UE8M0
 *    (power-of-two) scales.
 *  - "Where Rounding Happens Matters", section "the overall scheme": keep the
 *    intermediate in fp32 and round once at the end of a fused region (the
 *    GEMM's single bf16 rounding; here the reference result stays in fp64).
 *  - "MoE RL routing replay (R3)", section 4: fixed integer expert indices are
 *    replayed, so the grouped GEMM consumes fixed per-expert row segments.
 *
 * Readings where the pages are silent or garbled (each is listed in the
 * design notes of the repository):
 *  R1  scale = amax / 448 (IEEE fp32 division).  The page prints
 *      scale = max|W_block|, which would map every block into [-1, 1] and
 *      leave the E4M3 range unused; dividing by the format maximum 448 (the
 *      range printed on the same line) is the plain reading.
 *  R2  "round" is round-to-nearest, ties to even mantissa, saturating at
 *      +-448 (E4M3 has no infinity).  The sign of the result is the sign bit
 *      of the input, so -0 and negatives that round to zero give 0x80.
 *  R3  The value rounded to E4M3 is the fp32 quotient fl32(x / scale).
 *  R4  An all-zero block (amax == 0) stores scale 1.0 (UE8M0: exponent 0).
 *  R5  UE8M0 scale = 2^e with e the smallest integer such that
 *      448 * 2^e >= amax, clamped to [-127, 127], stored as the byte e + 127;
 *      the element is scaled by the exact power of two.
 *  R6  Activations use 1 x 128 groups along K (one scale per token and per
 *      128 columns); scales are stored K-group-major: scale[g][m].
 *  R7  Ragged edges: amax is taken over the valid elements of a partial
 *      block or group only.
 *  R12 Fused gate-up path (a "next" step: act-quant fused into the producing
 *      GEMM): the SwiGLU output SiLU(gate) * up is kept in fp32 (never rounded
 *      to bf16) and quantised in 1x128 groups by the same steps (R1-R6) as a
 *      bf16 activation; "Where Rounding Happens Matters", "the overall
 *      scheme".  The fp64 SiLU lives in the Python wrapper.
 *  R13 KV cache (a "next" step; "Method steps", step 3: the K/V quantisation
 *      scales are recomputed from the first forward of every RL step, before
 *      its rollout): one fp32 scale per tensor (the pages do not fix the
 *      granularity; per tensor is the plainest reading), scale = amax / 448
 *      of that calibration pass (R1, R4), and every K or V row written to the
 *      cache afterwards is quantised with it (R2, R3: values above the
 *      calibrated range saturate at +-448).  A slot index outside
 *      [0, num_slots) (padding) writes nothing.
 *
 * Everything is computed the plain way: decode and encode by explicit search
 * over the format's code table, fp64 dot products for the GEMM, no blocking.
 * Threads only split independent outer-loop iterations (blocks, groups,
 * output rows), which does not change any result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

enum { SCALE_FP32 = 0, SCALE_UE8M0 = 1 };

/* ------------------------------------------------------------------------ */
/* E4M3 format ("Prerequisites / FP8 quantisation format")                   */
/* ------------------------------------------------------------------------ */

/* Value of an E4M3 code from its bit fields: sign (1 bit), exponent (4 bits,
 * bias 7), mantissa (3 bits).  Exponent field 0 is subnormal: m * 2^-9.
 * The code with all exponent and mantissa bits set (0x7F / 0xFF) is NaN;
 * there is no infinity, so the largest finite magnitude is 0x7E. */
ORACLE_API double oracle_e4m3_decode(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* magnitudes of the 127 non-negative finite codes 0x00 .. 0x7E */
static double g_mag[127];
static pthread_once_t g_mag_once = PTHREAD_ONCE_INIT;

static void build_mag_table(void)
{
    for (int c = 0; c < 127; ++c)
        g_mag[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Saturating round-to-nearest-even of an exact value v into E4M3 (R2).
 * The 127 non-negative finite magnitudes increase strictly with the code, so
 * the search brackets |v| between two adjacent codes and compares against
 * their midpoint, which is exact in fp64. */
static uint8_t encode_value(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int lo, hi;
    pthread_once(&g_mag_once, build_mag_table);
    if (a >= g_mag[126]) /* 448 and beyond saturate */
        return sign | 126;
    lo = 0;
    hi = 126; /* invariant: g_mag[lo] <= a < g_mag[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_mag[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    {
        double midpoint = 0.5 * (g_mag[lo] + g_mag[hi]);
        int code;
        if (a < midpoint)
            code = lo;
        else if (a > midpoint)
            code = hi;
        else
            code = (lo & 1) ? hi : lo; /* tie: the code with even mantissa */
        return sign | (uint8_t)code;
    }
}

ORACLE_API uint8_t oracle_e4m3_encode(float v) { return encode_value((double)v); }

ORACLE_API uint8_t oracle_e4m3_encode_f64(double v) { return encode_value(v); }

/* ------------------------------------------------------------------------ */
/* bf16 input and the two scale formats                                      */
/* ------------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* R1 / R4: fp32 scale of a block or group with absolute maximum amax */
static float scale_fp32(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
    return amax / 448.0f;
}

/* R5: exponent of the UE8M0 scale */
static int scale_ue8m0_exponent(float amax)
{
    int e = -127;
    if (amax == 0.0f)
        return 0;
    while (e < 127 && ldexp(448.0, e) < (double)amax)
        ++e;
    return e;
}

ORACLE_API float oracle_scale_fp32(float amax) { return scale_fp32(amax); }

ORACLE_API int oracle_scale_ue8m0_exponent(float amax) { return scale_ue8m0_exponent(amax); }

/* value of a stored scale entry */
static double scale_value(const void* scales, int64_t idx, int fmt)
{
    if (fmt == SCALE_UE8M0)
        return ldexp(1.0, (int)((const uint8_t*)scales)[idx] - 127);
    return (double)((const float*)scales)[idx];
}

/* Quantise one rectangle of bf16 values (a weight block or an activation
 * group) with the given scale format; writes the codes and returns the stored
 * scale through *scale_f32 or *scale_u8. */
static void quantize_tile(const uint16_t* x, int64_t ldx, int64_t rows, int64_t cols,
                          uint8_t* q, int64_t ldq, int fmt, float* scale_f32, uint8_t* scale_u8)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(bf16_to_f32(x[r * ldx + c]));
            if (a > amax)
                amax = a;
        }
    if (fmt == SCALE_UE8M0) {
        int e = scale_ue8m0_exponent(amax);
        *scale_u8 = (uint8_t)(e + 127);
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c)
                q[r * ldq + c] = encode_value(ldexp((double)bf16_to_f32(x[r * ldx + c]), -e));
    } else {
        float scale = scale_fp32(amax);
        *scale_f32 = scale;
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c) {
                float quotient = bf16_to_f32(x[r * ldx + c]) / scale; /* R3 */
                q[r * ldq + c] = encode_value((double)quotient);
            }
    }
}

/* ------------------------------------------------------------------------ */
/* a tiny parallel-for over independent items                                */
/* ------------------------------------------------------------------------ */

typedef void (*item_fn)(void* ctx, int64_t item);

typedef struct {
    item_fn fn;
    void* ctx;
    int64_t count;
    int64_t begin, end;
} chunk_t;

static void* run_chunk(void* p)
{
    chunk_t* c = (chunk_t*)p;
    for (int64_t i = c->begin; i < c->end; ++i)
        c->fn(c->ctx, i);
    return NULL;
}

static void parallel_for(int64_t count, int threads, item_fn fn, void* ctx)
{
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if (threads == 1 || count < 2) {
        for (int64_t i = 0; i < count; ++i)
            fn(ctx, i);
        return;
    }
    {
        pthread_t tid[256];
        chunk_t chunk[256];
        int started[256];
        for (int t = 0; t < threads; ++t) {
            chunk[t].fn = fn;
            chunk[t].ctx = ctx;
            chunk[t].count = count;
            chunk[t].begin = count * t / threads;
            chunk[t].end = count * (t + 1) / threads;
            started[t] = pthread_create(&tid[t], NULL, run_chunk, &chunk[t]) == 0;
            if (!started[t])
                run_chunk(&chunk[t]);
        }
        for (int t = 0; t < threads; ++t)
            if (started[t])
                pthread_join(tid[t], NULL);
    }
}

/* ------------------------------------------------------------------------ */
/* Weight sync: 128x128 blockwise quantisation ("Method steps", step 1-2)     */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t* w;
    int64_t n, k, ldw;
    uint8_t* q;
    int64_t ldq;
    void* scale;
    int fmt;
    int64_t kb_count;
} wq_ctx;

static void wq_item(void* p, int64_t blk)
{
    wq_ctx* c = (wq_ctx*)p;
    int64_t nb = blk / c->kb_count, kb = blk % c->kb_count;
    int64_t r0 = nb * 128, c0 = kb * 128;
    int64_t rows = c->n - r0 < 128 ? c->n - r0 : 128; /* R7 */
    int64_t cols = c->k - c0 < 128 ? c->k - c0 : 128;
    float sf = 0.0f;
    uint8_t su = 0;
    quantize_tile(c->w + r0 * c->ldw + c0, c->ldw, rows, cols, c->q + r0 * c->ldq + c0, c->ldq,
                  c->fmt, &sf, &su);
    if (c->fmt == SCALE_UE8M0)
        ((uint8_t*)c->scale)[blk] = su;
    else
        ((float*)c->scale)[blk] = sf;
}

/* W: bf16 [n][k] (row stride ldw elements).  Q: E4M3 [n][k] (row stride ldq).
 * scale: [ceil(n/128)][ceil(k/128)] row-major, fp32 or UE8M0 bytes. */
ORACLE_API int oracle_quant_weight_blockwise(const uint16_t* w, int64_t n, int64_t k, int64_t ldw,
                                             uint8_t* q, int64_t ldq, void* scale, int fmt,
                                             int threads)
{
    wq_ctx c;
    if (n < 0 || k < 0 || ldw < k || ldq < k || (fmt != SCALE_FP32 && fmt != SCALE_UE8M0))
        return 1;
    c.w = w;
    c.n = n;
    c.k = k;
    c.ldw = ldw;
    c.q = q;
    c.ldq = ldq;
    c.scale = scale;
    c.fmt = fmt;
    c.kb_count = (k + 127) / 128;
    parallel_for(((n + 127) / 128) * c.kb_count, threads, wq_item, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Activations: dynamic 1x128 group quantisation (step 1, R6)                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t* x;
    int64_t m, k, ldx;
    uint8_t* q;
    int64_t ldq;
    void* scale;
    int fmt;
    int64_t groups;
} aq_ctx;

static void aq_item(void* p, int64_t row)
{
    aq_ctx* c = (aq_ctx*)p;
    for (int64_t g = 0; g < c->groups; ++g) {
        int64_t c0 = g * 128;
        int64_t cols = c->k - c0 < 128 ? c->k - c0 : 128;
        float sf = 0.0f;
        uint8_t su = 0;
        quantize_tile(c->x + row * c->ldx + c0, c->ldx, 1, cols, c->q + row * c->ldq + c0, c->ldq,
                      c->fmt, &sf, &su);
        if (c->fmt == SCALE_UE8M0)
            ((uint8_t*)c->scale)[g * c->m + row] = su;
        else
            ((float*)c->scale)[g * c->m + row] = sf;
    }
}

/* X: bf16 [m][k] (row stride ldx).  Q: E4M3 [m][k] (row stride ldq).
 * scale: [ceil(k/128)][m], fp32 or UE8M0 bytes. */
ORACLE_API int oracle_quant_act_group(const uint16_t* x, int64_t m, int64_t k, int64_t ldx,
                                      uint8_t* q, int64_t ldq, void* scale, int fmt, int threads)
{
    aq_ctx c;
    if (m < 0 || k < 0 || ldx < k || ldq < k || (fmt != SCALE_FP32 && fmt != SCALE_UE8M0))
        return 1;
    c.x = x;
    c.m = m;
    c.k = k;
    c.ldx = ldx;
    c.q = q;
    c.ldq = ldq;
    c.scale = scale;
    c.fmt = fmt;
    c.groups = (k + 127) / 128;
    parallel_for(m, threads, aq_item, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* fp32 activations: the same 1x128 group quantisation of values that were   */
/* never rounded to bf16 (the fused gate-up -> SwiGLU -> quantise path keeps  */
/* the SwiGLU output in fp32; "Where Rounding Happens Matters", "the overall  */
/* scheme").  Steps as above: amax over the group in fp32, R1/R4/R5 scale,   */
/* R3 fp32 quotient, R2 rounding.                                             */
/* ------------------------------------------------------------------------ */

static void quantize_group_f32(const float* x, int64_t cols, uint8_t* q, int fmt, float* scale_f32,
                               uint8_t* scale_u8)
{
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) {
        float a = fabsf(x[c]);
        if (a > amax)
            amax = a;
    }
    if (fmt == SCALE_UE8M0) {
        int e = scale_ue8m0_exponent(amax);
        *scale_u8 = (uint8_t)(e + 127);
        for (int64_t c = 0; c < cols; ++c)
            q[c] = encode_value(ldexp((double)x[c], -e));
    } else {
        float scale = scale_fp32(amax);
        *scale_f32 = scale;
        for (int64_t c = 0; c < cols; ++c) {
            float quotient = x[c] / scale; /* R3 */
            q[c] = encode_value((double)quotient);
        }
    }
}

typedef struct {
    const float* x;
    int64_t m, k, ldx;
    uint8_t* q;
    int64_t ldq;
    void* scale;
    int fmt;
    int64_t groups;
} aqf_ctx;

static void aqf_item(void* p, int64_t row)
{
    aqf_ctx* c = (aqf_ctx*)p;
    for (int64_t g = 0; g < c->groups; ++g) {
        int64_t c0 = g * 128;
        int64_t cols = c->k - c0 < 128 ? c->k - c0 : 128;
        float sf = 0.0f;
        uint8_t su = 0;
        quantize_group_f32(c->x + row * c->ldx + c0, cols, c->q + row * c->ldq + c0, c->fmt, &sf, &su);
        if (c->fmt == SCALE_UE8M0)
            ((uint8_t*)c->scale)[g * c->m + row] = su;
        else
            ((float*)c->scale)[g * c->m + row] = sf;
    }
}

/* X: fp32 [m][k] (row stride ldx).  Q: E4M3 [m][k] (row stride ldq).
 * scale: [ceil(k/128)][m], fp32 or UE8M0 bytes (R6 layout). */
ORACLE_API int oracle_quant_group_f32(const float* x, int64_t m, int64_t k, int64_t ldx, uint8_t* q,
                                      int64_t ldq, void* scale, int fmt, int threads)
{
    aqf_ctx c;
    if (m < 0 || k < 0 || ldx < k || ldq < k || (fmt != SCALE_FP32 && fmt != SCALE_UE8M0))
        return 1;
    c.x = x;
    c.m = m;
    c.k = k;
    c.ldx = ldx;
    c.q = q;
    c.ldq = ldq;
    c.scale = scale;
    c.fmt = fmt;
    c.groups = (k + 127) / 128;
    parallel_for(m, threads, aqf_item, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* KV cache: per-step per-tensor calibration and quantised append (R13)      */
/* ------------------------------------------------------------------------ */

static float tensor_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(bf16_to_f32(x[r * ld + c]));
            if (a > amax)
                amax = a;
        }
    return amax;
}

/* scales[0] = K scale, scales[1] = V scale, scales[2] = Q scale (q may be
 * null: scales[2] is left alone).  K and V are [tokens][kv_dim], Q is
 * [tokens][q_dim], bf16, with row strides ldk, ldv, ldq. */
ORACLE_API int oracle_kv_calibrate(const uint16_t* k, const uint16_t* v, const uint16_t* q, int64_t tokens,
                                   int64_t kv_dim, int64_t ldk, int64_t ldv, int64_t q_dim, int64_t ldq,
                                   float* scales)
{
    if (tokens < 0 || kv_dim < 0 || ldk < kv_dim || ldv < kv_dim || (q && (q_dim < 0 || ldq < q_dim)))
        return 1;
    scales[0] = scale_fp32(tensor_amax_bf16(k, tokens, kv_dim, ldk));
    scales[1] = scale_fp32(tensor_amax_bf16(v, tokens, kv_dim, ldv));
    if (q)
        scales[2] = scale_fp32(tensor_amax_bf16(q, tokens, q_dim, ldq));
    return 0;
}

/* Row t of K and V goes to cache row slots[t] (E4M3, row stride ldc) when
 * 0 <= slots[t] < num_slots; other cache rows are not touched. */
ORACLE_API int oracle_kv_append(const uint16_t* k, const uint16_t* v, int64_t tokens, int64_t kv_dim, int64_t ldk,
                                int64_t ldv, const int32_t* slots, uint8_t* k_cache, uint8_t* v_cache, int64_t ldc,
                                int64_t num_slots, const float* scales)
{
    if (tokens < 0 || kv_dim < 0 || ldk < kv_dim || ldv < kv_dim || ldc < kv_dim)
        return 1;
    for (int64_t t = 0; t < tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0 || slot >= num_slots)
            continue;
        for (int64_t c = 0; c < kv_dim; ++c) {
            float qk = bf16_to_f32(k[t * ldk + c]) / scales[0]; /* R3 */
            float qv = bf16_to_f32(v[t * ldv + c]) / scales[1];
            k_cache[slot * ldc + c] = encode_value((double)qk);
            v_cache[slot * ldc + c] = encode_value((double)qv);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Block-scaled W8A8 GEMM in fp64 ("compute-level W8A8")                     */
/*   Y[m][n] = sum_k (dec(qx[m][k]) * sx[k/128][m]) * (dec(qw[n][k]) * sw[n/128][k/128]) */
/* ------------------------------------------------------------------------ */

static double g_dec[256];
static pthread_once_t g_dec_once = PTHREAD_ONCE_INIT;

static void build_dec_table(void)
{
    for (int c = 0; c < 256; ++c)
        g_dec[c] = oracle_e4m3_decode((uint8_t)c);
}

/* one output element of the dequantised product; x_rows is the number of rows
 * the activation scale array was laid out for (its leading dimension) */
static double gemm_element(const uint8_t* xq, const void* sx, int64_t x_rows, const uint8_t* wq,
                           const void* sw, int64_t k, int fmt, int64_t row, int64_t col)
{
    int64_t kbs = k / 128;
    double acc = 0.0;
    for (int64_t kk = 0; kk < k; ++kk) {
        int64_t kb = kk / 128;
        double xv = g_dec[xq[row * k + kk]] * scale_value(sx, kb * x_rows + row, fmt);
        double wv = g_dec[wq[col * k + kk]] * scale_value(sw, (col / 128) * kbs + kb, fmt);
        acc += xv * wv;
    }
    return acc;
}

typedef struct {
    const uint8_t* xq;
    const void* sx;
    const uint8_t* wq;
    const void* sw;
    double* y;
    int64_t m, n, k;
    int fmt;
} gemm_ctx;

static void gemm_row(void* p, int64_t row)
{
    gemm_ctx* c = (gemm_ctx*)p;
    for (int64_t col = 0; col < c->n; ++col)
        c->y[row * c->n + col] = gemm_element(c->xq, c->sx, c->m, c->wq, c->sw, c->k, c->fmt, row, col);
}

/* xq E4M3 [m][k], sx [k/128][m], wq E4M3 [n][k], sw [n/128][k/128]; y fp64 [m][n].
 * n and k must be multiples of 128. */
ORACLE_API int oracle_gemm_blockscaled(const uint8_t* xq, const void* sx, const uint8_t* wq,
                                       const void* sw, double* y, int64_t m, int64_t n, int64_t k,
                                       int fmt, int threads)
{
    gemm_ctx c;
    if (m < 0 || n < 0 || k < 0 || n % 128 || k % 128 || (fmt != SCALE_FP32 && fmt != SCALE_UE8M0))
        return 1;
    pthread_once(&g_dec_once, build_dec_table);
    c.xq = xq;
    c.sx = sx;
    c.wq = wq;
    c.sw = sw;
    c.y = y;
    c.m = m;
    c.n = n;
    c.k = k;
    c.fmt = fmt;
    parallel_for(m, threads, gemm_row, &c);
    return 0;
}

typedef struct {
    const uint8_t* xq;
    const void* sx;
    const uint8_t* wq;
    const void* sw;
    int64_t m, n, k;
    int fmt;
    const int64_t* rows;
    const int64_t* cols;
    double* out;
} gemm_at_ctx;

static void gemm_at_item(void* p, int64_t i)
{
    gemm_at_ctx* c = (gemm_at_ctx*)p;
    c->out[i] = gemm_element(c->xq, c->sx, c->m, c->wq, c->sw, c->k, c->fmt, c->rows[i], c->cols[i]);
}

/* The same product evaluated only at the listed (row, col) positions. */
ORACLE_API int oracle_gemm_blockscaled_at(const uint8_t* xq, const void* sx, const uint8_t* wq,
                                          const void* sw, int64_t m, int64_t n, int64_t k, int fmt,
                                          const int64_t* rows, const int64_t* cols, int64_t count,
                                          double* out, int threads)
{
    gemm_at_ctx c;
    if (m < 0 || n < 0 || k < 0 || n % 128 || k % 128 || (fmt != SCALE_FP32 && fmt != SCALE_UE8M0))
        return 1;
    for (int64_t i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= m || cols[i] < 0 || cols[i] >= n)
            return 2;
    pthread_once(&g_dec_once, build_dec_table);
    c.xq = xq;
    c.sx = sx;
    c.wq = wq;
    c.sw = sw;
    c.m = m;
    c.n = n;
    c.k = k;
    c.fmt = fmt;
    c.rows = rows;
    c.cols = cols;
    c.out = out;
    parallel_for(count, threads, gemm_at_item, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped (MoE expert) GEMM: rows offsets[e] .. offsets[e+1]-1 use expert e  */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* xq;
    const void* sx;
    const uint8_t* wq;
    const void* sw;
    const int32_t* offsets;
    int64_t experts, rows, n, k;
    int fmt;
    const int64_t* at_rows;
    const int64_t* at_cols;
    double* out;
    double* y;
} grouped_ctx;

static int64_t expert_of_row(const int32_t* offsets, int64_t experts, int64_t row)
{
    /* the expert whose segment [offsets[e], offsets[e+1]) holds row */
    for (int64_t e = 0; e < experts; ++e)
        if (row >= offsets[e] && row < offsets[e + 1])
            return e;
    return -1;
}

static double grouped_element(const grouped_ctx* c, int64_t row, int64_t col)
{
    int64_t e = expert_of_row(c->offsets, c->experts, row);
    int64_t wsz = c->n * c->k;
    int64_t ssz = (c->n / 128) * (c->k / 128);
    size_t sbytes = c->fmt == SCALE_UE8M0 ? 1 : 4;
    if (e < 0)
        return 0.0;
    return gemm_element(c->xq, c->sx, c->rows, c->wq + e * wsz, (const char*)c->sw + e * ssz * sbytes,
                        c->k, c->fmt, row, col);
}

static void grouped_row(void* p, int64_t row)
{
    grouped_ctx* c = (grouped_ctx*)p;
    for (int64_t col = 0; col < c->n; ++col)
        c->y[row * c->n + col] = grouped_element(c, row, col);
}

static void grouped_at_item(void* p, int64_t i)
{
    grouped_ctx* c = (grouped_ctx*)p;
    c->out[i] = grouped_element(c, c->at_rows[i], c->at_cols[i]);
}

static int grouped_check(const int32_t* offsets, int64_t experts, int64_t rows, int64_t n, int64_t k,
                         int fmt)
{
    if (experts < 1 || rows < 0 || n < 0 || k < 0 || n % 128 || k % 128)
        return 1;
    if (fmt != SCALE_FP32 && fmt != SCALE_UE8M0)
        return 1;
    if (offsets[0] != 0 || offsets[experts] != rows)
        return 3;
    for (int64_t e = 0; e < experts; ++e)
        if (offsets[e + 1] < offsets[e])
            return 3;
    return 0;
}

/* xq [rows][k], sx [k/128][rows], wq [experts][n][k], sw [experts][n/128][k/128],
 * offsets int32 [experts+1] (host memory), y fp64 [rows][n]. */
ORACLE_API int oracle_grouped_gemm_blockscaled(const uint8_t* xq, const void* sx, const uint8_t* wq,
                                               const void* sw, const int32_t* offsets, int64_t experts,
                                               int64_t rows, int64_t n, int64_t k, double* y, int fmt,
                                               int threads)
{
    grouped_ctx c;
    int rc = grouped_check(offsets, experts, rows, n, k, fmt);
    if (rc)
        return rc;
    pthread_once(&g_dec_once, build_dec_table);
    memset(&c, 0, sizeof c);
    c.xq = xq;
    c.sx = sx;
    c.wq = wq;
    c.sw = sw;
    c.offsets = offsets;
    c.experts = experts;
    c.rows = rows;
    c.n = n;
    c.k = k;
    c.fmt = fmt;
    c.y = y;
    parallel_for(rows, threads, grouped_row, &c);
    return 0;
}

ORACLE_API int oracle_grouped_gemm_blockscaled_at(const uint8_t* xq, const void* sx, const uint8_t* wq,
                                                  const void* sw, const int32_t* offsets,
                                                  int64_t experts, int64_t rows, int64_t n, int64_t k,
                                                  int fmt, const int64_t* at_rows,
                                                  const int64_t* at_cols, int64_t count, double* out,
                                                  int threads)
{
    grouped_ctx c;
    int rc = grouped_check(offsets, experts, rows, n, k, fmt);
    if (rc)
        return rc;
    for (int64_t i = 0; i < count; ++i)
        if (at_rows[i] < 0 || at_rows[i] >= rows || at_cols[i] < 0 || at_cols[i] >= n)
            return 2;
    pthread_once(&g_dec_once, build_dec_table);
    memset(&c, 0, sizeof c);
    c.xq = xq;
    c.sx = sx;
    c.wq = wq;
    c.sw = sw;
    c.offsets = offsets;
    c.experts = experts;
    c.rows = rows;
    c.n = n;
    c.k = k;
    c.fmt = fmt;
    c.at_rows = at_rows;
    c.at_cols = at_cols;
    c.out = out;
    parallel_for(count, threads, grouped_at_item, &c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* bulk encode (for whole-format checks of a device codec)                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    const float* v;
    uint8_t* out;
    int64_t n;
    int64_t chunk;
} enc_ctx;

static void enc_item(void* p, int64_t i)
{
    enc_ctx* c = (enc_ctx*)p;
    int64_t b = i * c->chunk, e = b + c->chunk < c->n ? b + c->chunk : c->n;
    for (int64_t j = b; j < e; ++j)
        c->out[j] = encode_value((double)c->v[j]);
}

ORACLE_API void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out, int threads)
{
    enc_ctx c;
    c.v = v;
    c.out = out;
    c.n = n;
    c.chunk = 1 << 16;
    parallel_for((n + c.chunk - 1) / c.chunk, threads, enc_item, &c);
}
