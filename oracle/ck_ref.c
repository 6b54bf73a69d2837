/*
 * ck_ref.c -- the oracle: a plain, slow, scalar CPU statement of the
 * single-token attention decode step with Q5_0 / Q8_0 weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only in the bytes of their inputs and outputs.
 *
 * Source of every step: the page "mega_fused_attention_decode_q5_0.c"
 * (C-Kernel-Engine doxygen), whose serial kernel is the composition
 *   RMSNorm -> Q8_0 quantize -> Q/K (Q5_0) and V (Q8_0) GEMV + bias -> RoPE
 *   -> KV-cache store -> GQA decode attention -> Q8_0 quantize -> O (Q5_0)
 *   GEMV + bias + residual.
 * The page declares but does not print rmsnorm_forward, quantize_row_q8_0,
 * the vec_dot routines and the attention routine; the readings taken for
 * them are stated beside each function below.
 *
 * Precision: every reduction is carried in double and rounded once to fp32,
 * so the oracle is the exact result up to one final rounding wherever that
 * is cheap to state.  Compile with -ffp-contract=off and without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Block sizes of the two formats (page: QK5_0 / QK8_0 blocks of 32). */
#define REF_QK 32
#define REF_Q5_0_BYTES 22 /* fp16 d, u32 qh, 16 bytes of nibbles */
#define REF_Q8_0_BYTES 34 /* fp16 d, 32 int8 */

/* ------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary32, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have
 * exponent field 0 and value frac * 2^-24.  Conversion to binary16 rounds
 * to nearest, ties to even, and overflows to infinity.
 * ---------------------------------------------------------------------- */
float ref_f16_to_f32(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + f), e - 25);
    return sign ? -v : v;
}

uint16_t ref_f32_to_f16(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    const uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    const uint32_t a = b & 0x7fffffffu;
    if (a >= 0x7f800000u) /* inf or nan */
        return sign | (a > 0x7f800000u ? 0x7e00u : 0x7c00u);
    const int fexp = (int)(a >> 23);
    if (fexp == 0) /* fp32 subnormal: far below half of the smallest half */
        return sign;
    const int E = fexp - 127;                       /* x = m * 2^(E-23) */
    if (E > 15)
        return sign | 0x7c00u;
    if (E < -25)
        return sign;
    const uint32_t m = (a & 0x7fffffu) | 0x800000u; /* 24-bit significand */
    /* exponent of one unit in the last place of the binary16 result */
    const int ulp_e = (E >= -14) ? E - 10 : -24;
    const int shift = 23 + ulp_e - E;               /* 13 .. 24 */
    uint32_t q = m >> shift;
    const uint32_t rem = m & ((1u << shift) - 1u);
    const uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q++;
    if (E >= -14) /* normal: q in [1024, 2048]; a carry moves the exponent */
        return sign | (uint16_t)((uint32_t)(E + 15) * 1024u + q - 1024u);
    return sign | (uint16_t)q; /* subnormal (q == 1024 is the smallest normal) */
}

/* Array forms of the two conversions (used by the codec self-checks). */
void ref_f32_to_f16_n(const float *x, uint16_t *h, long n)
{
    for (long i = 0; i < n; ++i)
        h[i] = ref_f32_to_f16(x[i]);
}

void ref_f16_to_f32_n(const uint16_t *h, float *x, long n)
{
    for (long i = 0; i < n; ++i)
        x[i] = ref_f16_to_f32(h[i]);
}

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t rd_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* ------------------------------------------------------------------------
 * Block codecs.  Byte layout (the pages give only the field list; this is
 * the reading): Q5_0 = d (fp16, little-endian) at byte 0, qh (u32 LE) at
 * byte 2, qs[16] at byte 6; element j < 16 has low nibble qs[j] & 15 and
 * high bit (qh >> j) & 1, element j + 16 has qs[j] >> 4 and bit j + 16;
 * code q in [0, 31], weight (q - 16) * d.  Q8_0 = d at byte 0, int8 qs[32]
 * at byte 2, weight q * d.
 * ---------------------------------------------------------------------- */
void ref_unpack_q5_0(const uint8_t *blk, int32_t *q, float *d)
{
    const uint32_t qh = rd_u32(blk + 2);
    for (int j = 0; j < 16; ++j) {
        const int lo = blk[6 + j] & 0x0f;
        const int hi = blk[6 + j] >> 4;
        q[j] = (lo | (int)(((qh >> j) & 1u) << 4)) - 16;
        q[j + 16] = (hi | (int)(((qh >> (j + 16)) & 1u) << 4)) - 16;
    }
    *d = ref_f16_to_f32(rd_u16(blk));
}

void ref_unpack_q8_0(const uint8_t *blk, int32_t *q, float *d)
{
    for (int j = 0; j < REF_QK; ++j)
        q[j] = (int8_t)blk[2 + j];
    *d = ref_f16_to_f32(rd_u16(blk));
}

void ref_dequant_q5_0(const uint8_t *blk, float *w)
{
    int32_t q[REF_QK];
    float d;
    ref_unpack_q5_0(blk, q, &d);
    for (int j = 0; j < REF_QK; ++j)
        w[j] = (float)((double)q[j] * (double)d);
}

void ref_dequant_q8_0(const uint8_t *blk, float *w)
{
    int32_t q[REF_QK];
    float d;
    ref_unpack_q8_0(blk, q, &d);
    for (int j = 0; j < REF_QK; ++j)
        w[j] = (float)((double)q[j] * (double)d);
}

/* ------------------------------------------------------------------------
 * quantize_row_q8_0 (declared on the page, body not shown).  Reading, per
 * block of 32: amax = max |x_i|; d = amax / 127 in fp32; id = 1/d (0 when
 * d == 0); q_i = round-half-away-from-zero(x_i * id); d is stored as fp16.
 * ---------------------------------------------------------------------- */
void ref_quantize_row_q8_0(const float *x, uint8_t *y, int n)
{
    for (int b = 0; b < n / REF_QK; ++b) {
        const float *xb = x + (size_t)b * REF_QK;
        uint8_t *yb = y + (size_t)b * REF_Q8_0_BYTES;
        float amax = 0.0f;
        for (int j = 0; j < REF_QK; ++j) {
            const float a = fabsf(xb[j]);
            if (a > amax)
                amax = a;
        }
        const float d = amax / 127.0f;
        const float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        const uint16_t dh = ref_f32_to_f16(d);
        yb[0] = (uint8_t)(dh & 0xff);
        yb[1] = (uint8_t)(dh >> 8);
        for (int j = 0; j < REF_QK; ++j) {
            const float v = xb[j] * id;
            yb[2 + j] = (uint8_t)(int8_t)(int)roundf(v);
        }
    }
}

/* ------------------------------------------------------------------------
 * vec_dot_q5_0_q8_0 / vec_dot_q8_0_q8_0, per block: the integer dot of the
 * two code vectors, exact in int32.
 * ---------------------------------------------------------------------- */
int32_t ref_block_dot_q5_0_q8_0(const uint8_t *w, const uint8_t *x)
{
    int32_t qw[REF_QK], qx[REF_QK];
    float dw, dx;
    ref_unpack_q5_0(w, qw, &dw);
    ref_unpack_q8_0(x, qx, &dx);
    int32_t s = 0;
    for (int j = 0; j < REF_QK; ++j)
        s += qw[j] * qx[j];
    return s;
}

int32_t ref_block_dot_q8_0_q8_0(const uint8_t *w, const uint8_t *x)
{
    int32_t qw[REF_QK], qx[REF_QK];
    float dw, dx;
    ref_unpack_q8_0(w, qw, &dw);
    ref_unpack_q8_0(x, qx, &dx);
    int32_t s = 0;
    for (int j = 0; j < REF_QK; ++j)
        s += qw[j] * qx[j];
    return s;
}

/* Per-block integer dots of every row of W against x: isum[M, K/32]. */
void ref_block_dots(int32_t *isum, const uint8_t *W, const uint8_t *xq, int M, int K, int w_is_q8)
{
    const int nb = K / REF_QK;
    const int wb = w_is_q8 ? REF_Q8_0_BYTES : REF_Q5_0_BYTES;
    for (int r = 0; r < M; ++r)
        for (int b = 0; b < nb; ++b) {
            const uint8_t *w = W + ((size_t)r * nb + b) * wb;
            const uint8_t *x = xq + (size_t)b * REF_Q8_0_BYTES;
            isum[(size_t)r * nb + b] = w_is_q8 ? ref_block_dot_q8_0_q8_0(w, x) : ref_block_dot_q5_0_q8_0(w, x);
        }
}

/* ------------------------------------------------------------------------
 * gemv_q5_0_from_fp32 / gemv_q8_0_from_fp32 after the activation has been
 * quantized: out[r] = dot(W[r], x) + bias[r] (bias may be NULL), where the
 * dot is sum_b d_w(b) * d_x(b) * isum(b).  Each block term is exact in
 * double; the row sum is rounded once to fp32 and the bias added in fp32.
 * ---------------------------------------------------------------------- */
void ref_gemv(float *y, const uint8_t *W, const uint8_t *xq, const float *bias, int M, int K, int w_is_q8)
{
    const int nb = K / REF_QK;
    const int wb = w_is_q8 ? REF_Q8_0_BYTES : REF_Q5_0_BYTES;
    for (int r = 0; r < M; ++r) {
        double acc = 0.0;
        for (int b = 0; b < nb; ++b) {
            const uint8_t *w = W + ((size_t)r * nb + b) * wb;
            const uint8_t *x = xq + (size_t)b * REF_Q8_0_BYTES;
            const int32_t s = w_is_q8 ? ref_block_dot_q8_0_q8_0(w, x) : ref_block_dot_q5_0_q8_0(w, x);
            const double dw = ref_f16_to_f32(rd_u16(w));
            const double dx = ref_f16_to_f32(rd_u16(x));
            acc += dw * dx * (double)s;
        }
        const float dot = (float)acc;
        y[r] = dot + (bias ? bias[r] : 0.0f);
    }
}

/* ------------------------------------------------------------------------
 * rmsnorm_forward for one token over all D elements (the page calls it with
 * T = 1 and D = the aligned embed dim).  Reading: rstd = 1/sqrt(mean(x^2)
 * + eps) with the mean in double, rounded to fp32; y_i = (x_i * rstd) *
 * gamma_i, two fp32 multiplies.
 * ---------------------------------------------------------------------- */
float ref_rmsnorm(const float *x, const float *gamma, float *y, int D, float eps)
{
    double ss = 0.0;
    for (int i = 0; i < D; ++i)
        ss += (double)x[i] * (double)x[i];
    const float rstd = (float)(1.0 / sqrt(ss / (double)D + (double)eps));
    for (int i = 0; i < D; ++i) {
        const float t = x[i] * rstd;
        y[i] = t * gamma[i];
    }
    return rstd;
}

/* ------------------------------------------------------------------------
 * apply_rope_inline: rotate-half RoPE.  With half = hd/2 and table row
 * `pos` of cos/sin [capacity, half], element d pairs with d + half:
 *   a' = a*cos - b*sin,  b' = a*sin + b*cos,
 * for every query head and every key head; V is not rotated.
 * ---------------------------------------------------------------------- */
static void rope_heads(float *v, int heads, int hd, const float *c, const float *s)
{
    const int half = hd / 2;
    for (int h = 0; h < heads; ++h) {
        float *p = v + (size_t)h * hd;
        for (int d = 0; d < half; ++d) {
            const float a = p[d];
            const float b = p[d + half];
            const float ac = a * c[d], bs = b * s[d];
            const float as = a * s[d], bc = b * c[d];
            p[d] = ac - bs;
            p[d + half] = as + bc;
        }
    }
}

void ref_rope(float *q, float *k, const float *rope_cos, const float *rope_sin, int pos, int H, int KV, int hd)
{
    const float *c = rope_cos + (size_t)pos * (hd / 2);
    const float *s = rope_sin + (size_t)pos * (hd / 2);
    if (q)
        rope_heads(q, H, hd, c, s);
    if (k)
        rope_heads(k, KV, hd, c, s);
}

/* KV-cache store: caches are head-major [KV, capacity, hd]; row `pos` of
 * each KV head receives that head's rotated K and its V. */
void ref_kv_store(float *k_cache, float *v_cache, const float *k, const float *v, int pos, int KV, int capacity, int hd)
{
    for (int h = 0; h < KV; ++h) {
        const size_t off = ((size_t)h * capacity + (size_t)pos) * hd;
        for (int d = 0; d < hd; ++d) {
            k_cache[off + d] = k[(size_t)h * hd + d];
            v_cache[off + d] = v[(size_t)h * hd + d];
        }
    }
}

/* ------------------------------------------------------------------------
 * attention_forward_decode_head_major_gqa_flash (declared on the page; body
 * not shown).  Query head h reads KV head h*KV/H; for the kv_tokens cache
 * rows t: s_t = (q_h . k_t) / sqrt(hd); out_h = sum_t softmax(s)_t v_t.
 * Stated here as the plain two-pass softmax in double.
 * ---------------------------------------------------------------------- */
void ref_attention(const float *q, const float *k_cache, const float *v_cache, float *out, int H, int KV, int T,
                   int capacity, int hd)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)hd);
    const double scale = 1.0 / sqrt((double)hd);
    for (int h = 0; h < H; ++h) {
        const int kvh = (int)((long)h * KV / H);
        const float *qh = q + (size_t)h * hd;
        const float *kb = k_cache + (size_t)kvh * capacity * hd;
        const float *vb = v_cache + (size_t)kvh * capacity * hd;
        double m = -INFINITY;
        for (int t = 0; t < T; ++t) {
            double dot = 0.0;
            for (int d = 0; d < hd; ++d)
                dot += (double)qh[d] * (double)kb[(size_t)t * hd + d];
            s[t] = dot * scale;
            if (s[t] > m)
                m = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < T; ++t) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        for (int d = 0; d < hd; ++d)
            o[d] = 0.0;
        for (int t = 0; t < T; ++t)
            for (int d = 0; d < hd; ++d)
                o[d] += s[t] * (double)vb[(size_t)t * hd + d];
        for (int d = 0; d < hd; ++d)
            out[(size_t)h * hd + d] = (float)(o[d] / l);
    }
    free(s);
    free(o);
}

/* ------------------------------------------------------------------------
 * Reduced-precision KV caches (page "prefill_attn_a.rs", layers/ops:
 * the launchers paged_decode_attn_bf16 / paged_decode_attn_fp8: bf16 and fp8 caches, the
 * fp8 one with per-tensor k_scale and v_scale; the pages print only the
 * launchers, so the element formats are taken from their definitions):
 *
 * bfloat16: the upper 16 bits of a binary32 (1 sign, 8 exponent, 7 fraction
 *   bits).  From binary32: round to nearest, ties to even (a NaN stays NaN).
 * E4M3 ("FN" 8-bit float): 1 sign, 4 exponent bits with bias 7, 3 fraction
 *   bits; exponent field 0 holds subnormals frac * 2^-9; S.1111.111 is NaN;
 *   no infinity; the largest finite magnitude is 1.75 * 2^8 = 448.  From
 *   binary32: round to nearest, ties to even, magnitudes beyond 448
 *   saturate to 448, NaN gives NaN.
 * The cache value is the bf16 number, or code * k_scale (keys) and
 * code * v_scale (values) for E4M3.  A store quantizes x / scale (the IEEE
 * binary32 quotient).
 * ---------------------------------------------------------------------- */
float ref_bf16_to_f32(uint16_t b)
{
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t ref_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t t = u >> 16;           /* truncated: the representable value toward zero */
    const uint32_t r = u & 0xFFFFu; /* the discarded bits */
    if (r > 0x8000u || (r == 0x8000u && (t & 1u)))
        t += 1u; /* the next magnitude up (into the exponent, or to infinity) */
    return (uint16_t)t;
}

float ref_e4m3_to_f32(uint8_t c)
{
    const int e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* (m / 8) * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 10); /* (1 + m / 8) * 2^(e - 7) */
    return (float)((c & 0x80) ? -v : v);
}

uint8_t ref_f32_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7F;
    const int sign = signbit(x) ? 0x80 : 0;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* the nearest of the non-negative finite codes 0x00 .. 0x7E (values
     * increase with the code); on a tie, the even code */
    int best = 0;
    double bd = a;
    for (int c = 1; c <= 0x7E; ++c) {
        const double d = fabs((double)ref_e4m3_to_f32((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    return (uint8_t)(sign | best);
}

void ref_f32_to_bf16_n(const float *x, uint16_t *y, long n)
{
    for (long i = 0; i < n; ++i)
        y[i] = ref_f32_to_bf16(x[i]);
}

/* codes of x / scale (binary32 quotients) */
void ref_f32_to_e4m3_n(const float *x, float scale, uint8_t *y, long n)
{
    for (long i = 0; i < n; ++i)
        y[i] = ref_f32_to_e4m3(x[i] / scale);
}

void ref_e4m3_to_f32_n(const uint8_t *c, float *y, long n)
{
    for (long i = 0; i < n; ++i)
        y[i] = ref_e4m3_to_f32(c[i]);
}

/* value of element i of a reduced cache: kind 1 = bf16, 2 = E4M3 * scale */
static double kvq_value(const void *cache, size_t i, int kind, double scale)
{
    if (kind == 1)
        return (double)ref_bf16_to_f32(((const uint16_t *)cache)[i]);
    return (double)ref_e4m3_to_f32(((const uint8_t *)cache)[i]) * scale;
}

/* ref_attention over a bf16 (kind 1) or E4M3 (kind 2) cache: the same
 * two-pass softmax in double on the caches' values. */
void ref_attention_kvq(const float *q, const void *k_cache, const void *v_cache, float *out, int H, int KV, int T,
                       int capacity, int hd, int kind, float k_scale, float v_scale)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)hd);
    const double scale = 1.0 / sqrt((double)hd);
    for (int h = 0; h < H; ++h) {
        const int kvh = (int)((long)h * KV / H);
        const float *qh = q + (size_t)h * hd;
        const size_t base = (size_t)kvh * capacity * hd;
        double m = -INFINITY;
        for (int t = 0; t < T; ++t) {
            double dot = 0.0;
            for (int d = 0; d < hd; ++d)
                dot += (double)qh[d] * kvq_value(k_cache, base + (size_t)t * hd + d, kind, k_scale);
            s[t] = dot * scale;
            if (s[t] > m)
                m = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < T; ++t) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        for (int d = 0; d < hd; ++d)
            o[d] = 0.0;
        for (int t = 0; t < T; ++t)
            for (int d = 0; d < hd; ++d)
                o[d] += s[t] * kvq_value(v_cache, base + (size_t)t * hd + d, kind, v_scale);
        for (int d = 0; d < hd; ++d)
            out[(size_t)h * hd + d] = (float)(o[d] / l);
    }
    free(s);
    free(o);
}

/* STEP 6 into a reduced cache: row pos of every KV head. */
void ref_kv_store_kvq(void *k_cache, void *v_cache, const float *k, const float *v, int pos, int KV, int capacity,
                      int hd, int kind, float k_scale, float v_scale)
{
    for (int h = 0; h < KV; ++h)
        for (int d = 0; d < hd; ++d) {
            const size_t i = ((size_t)h * capacity + pos) * hd + d, j = (size_t)h * hd + d;
            if (kind == 1) {
                ((uint16_t *)k_cache)[i] = ref_f32_to_bf16(k[j]);
                ((uint16_t *)v_cache)[i] = ref_f32_to_bf16(v[j]);
            } else {
                ((uint8_t *)k_cache)[i] = ref_f32_to_e4m3(k[j] / k_scale);
                ((uint8_t *)v_cache)[i] = ref_f32_to_e4m3(v[j] / v_scale);
            }
        }
}

/* ------------------------------------------------------------------------
 * Paged decode attention with a sliding window (page
 * "prefill_attn_a.rs", layers/ops: paged_decode_attn_bf16 / _fp8 and their GQA forms; only the
 * launchers are printed).  Readings: the pools are [num_blocks][KV]
 * [block_size][hd]; row t of sequence b is row t % block_size of physical
 * block block_tables[b * max_blocks + t / block_size]; the sequence attends
 * rows [T0, T) with T = seq_lens[b] and T0 = max(0, T - window) when
 * window > 0, else 0; the attention is ref_attention's on those rows.
 * kind: 0 fp32, 1 bf16, 2 E4M3 (values as in ref_attention_kvq).
 * ---------------------------------------------------------------------- */
static double pool_value(const void *pool, size_t i, int kind, double scale)
{
    if (kind == 0)
        return (double)((const float *)pool)[i];
    return kvq_value(pool, i, kind, scale);
}

void ref_attention_paged(const float *q, const void *k_pool, const void *v_pool, float *out,
                         const int32_t *block_tables, const int32_t *seq_lens, int B, int H, int KV, int hd,
                         int block_size, int max_blocks, int window, int kind, float k_scale, float v_scale)
{
    const double scale = 1.0 / sqrt((double)hd);
    for (int b = 0; b < B; ++b) {
        const int T = seq_lens[b];
        const int T0 = (window > 0 && T > window) ? T - window : 0;
        const int n = T - T0;
        double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)hd);
        for (int h = 0; h < H; ++h) {
            const int kvh = (int)((long)h * KV / H);
            const float *qh = q + ((size_t)b * H + h) * hd;
            double m = -INFINITY;
            for (int t = T0; t < T; ++t) {
                const int pb = block_tables[(size_t)b * max_blocks + t / block_size];
                const size_t base = (((size_t)pb * KV + kvh) * block_size + t % block_size) * hd;
                double dot = 0.0;
                for (int d = 0; d < hd; ++d)
                    dot += (double)qh[d] * pool_value(k_pool, base + d, kind, k_scale);
                s[t - T0] = dot * scale;
                if (s[t - T0] > m)
                    m = s[t - T0];
            }
            double l = 0.0;
            for (int i = 0; i < n; ++i) {
                s[i] = exp(s[i] - m);
                l += s[i];
            }
            for (int d = 0; d < hd; ++d)
                o[d] = 0.0;
            for (int t = T0; t < T; ++t) {
                const int pb = block_tables[(size_t)b * max_blocks + t / block_size];
                const size_t base = (((size_t)pb * KV + kvh) * block_size + t % block_size) * hd;
                for (int d = 0; d < hd; ++d)
                    o[d] += s[t - T0] * pool_value(v_pool, base + d, kind, v_scale);
            }
            for (int d = 0; d < hd; ++d)
                out[((size_t)b * H + h) * hd + d] = n > 0 ? (float)(o[d] / l) : 0.0f;
        }
        free(s);
        free(o);
    }
}

/* ------------------------------------------------------------------------
 * mega_fused_attention_decode_q5_0, in the page's order (STEP 1 .. STEP 8).
 * `dbg_*` are optional (NULL-able) taps of the intermediates:
 *   dbg_xq   [D/32 Q8_0 blocks]   the quantized normed input
 *   dbg_q    [H*hd]               q after bias and RoPE
 *   dbg_k    [KV*hd]              k after bias and RoPE (= stored row)
 *   dbg_v    [KV*hd]              v after bias (= stored row)
 *   dbg_attn [H*hd]               attention output
 *   dbg_aq   [H*hd/32 blocks]     the quantized attention output
 * ---------------------------------------------------------------------- */
void ref_decode_layer(float *out, const float *x, const float *residual, const uint8_t *wq, const uint8_t *wk,
                      const uint8_t *wv, const uint8_t *wo, const float *gamma, const float *bq, const float *bk,
                      const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                      const float *rope_sin, int pos, int D, int H, int KV, int hd, int capacity, float eps,
                      uint8_t *dbg_xq, float *dbg_q, float *dbg_k, float *dbg_v, float *dbg_attn, uint8_t *dbg_aq)
{
    const int QD = H * hd, KD = KV * hd;
    float *xn = (float *)malloc(sizeof(float) * (size_t)D);
    float *q = (float *)malloc(sizeof(float) * (size_t)QD);
    float *k = (float *)malloc(sizeof(float) * (size_t)KD);
    float *v = (float *)malloc(sizeof(float) * (size_t)KD);
    float *attn = (float *)malloc(sizeof(float) * (size_t)QD);
    const int maxd = D > QD ? D : QD;
    uint8_t *xq = (uint8_t *)malloc((size_t)(maxd / REF_QK) * REF_Q8_0_BYTES);

    /* 1: RMSNorm */
    ref_rmsnorm(x, gamma, xn, D, eps);
    /* 2-4: Q, K (Q5_0) and V (Q8_0) projections on the Q8_0 activation */
    ref_quantize_row_q8_0(xn, xq, D);
    if (dbg_xq)
        memcpy(dbg_xq, xq, (size_t)(D / REF_QK) * REF_Q8_0_BYTES);
    ref_gemv(q, wq, xq, bq, QD, D, 0);
    ref_gemv(k, wk, xq, bk, KD, D, 0);
    ref_gemv(v, wv, xq, bv, KD, D, 1);
    /* 5: RoPE */
    ref_rope(q, k, rope_cos, rope_sin, pos, H, KV, hd);
    /* 6: KV-cache store */
    ref_kv_store(k_cache, v_cache, k, v, pos, KV, capacity, hd);
    /* 7: attention over pos + 1 rows */
    ref_attention(q, k_cache, v_cache, attn, H, KV, pos + 1, capacity, hd);
    /* 8: O projection + bias + residual */
    ref_quantize_row_q8_0(attn, xq, QD);
    if (dbg_aq)
        memcpy(dbg_aq, xq, (size_t)(QD / REF_QK) * REF_Q8_0_BYTES);
    ref_gemv(out, wo, xq, bo, D, QD, 0);
    for (int e = 0; e < D; ++e)
        out[e] = out[e] + residual[e];

    if (dbg_q)
        memcpy(dbg_q, q, sizeof(float) * (size_t)QD);
    if (dbg_k)
        memcpy(dbg_k, k, sizeof(float) * (size_t)KD);
    if (dbg_v)
        memcpy(dbg_v, v, sizeof(float) * (size_t)KD);
    if (dbg_attn)
        memcpy(dbg_attn, attn, sizeof(float) * (size_t)QD);
    free(xn);
    free(q);
    free(k);
    free(v);
    free(attn);
    free(xq);
}

/* ------------------------------------------------------------------------
 * The multi-token (prefill) form of the same layer: n tokens of ONE sequence,
 * token i at position pos + i, causal.  Page "prefill_attn_a.rs"
 * (layers/ops), the prefill attention launcher: one query per (head, token)
 * with a causal switch; read here as token i attending cache rows
 * 0 .. pos + i, i.e. the rows already in the cache plus the chunk's own rows
 * up to and including its own.
 *
 * The plain definition, in two phases: STEP 1 .. STEP 6 of the decode layer
 * (norm, Q8_0 quant, projections, RoPE at pos + i, KV store at row pos + i)
 * for every token, then STEP 7 .. STEP 8 (attention over pos + i + 1 rows,
 * quant, O projection, residual) for every token.  x, residual, out:
 * fp32 [n][D].  Taps as for ref_decode_layer, each [n][...] (NULL-able).
 * ---------------------------------------------------------------------- */
void ref_prefill_layer(float *out, const float *x, const float *residual, const uint8_t *wq, const uint8_t *wk,
                       const uint8_t *wv, const uint8_t *wo, const float *gamma, const float *bq, const float *bk,
                       const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                       const float *rope_sin, int pos, int n, int D, int H, int KV, int hd, int capacity, float eps,
                       uint8_t *dbg_xq, float *dbg_q, float *dbg_k, float *dbg_v, float *dbg_attn, uint8_t *dbg_aq)
{
    const int QD = H * hd, KD = KV * hd;
    const size_t xq_bytes = (size_t)(D / REF_QK) * REF_Q8_0_BYTES;
    const size_t aq_bytes = (size_t)(QD / REF_QK) * REF_Q8_0_BYTES;
    float *xn = (float *)malloc(sizeof(float) * (size_t)D);
    float *q = (float *)malloc(sizeof(float) * (size_t)QD * (size_t)n);
    float *k = (float *)malloc(sizeof(float) * (size_t)KD);
    float *v = (float *)malloc(sizeof(float) * (size_t)KD);
    float *attn = (float *)malloc(sizeof(float) * (size_t)QD);
    uint8_t *xq = (uint8_t *)malloc(xq_bytes > aq_bytes ? xq_bytes : aq_bytes);

    /* phase 1: every token's q, and its k / v stored at row pos + i */
    for (int i = 0; i < n; ++i) {
        float *qi = q + (size_t)i * QD;
        ref_rmsnorm(x + (size_t)i * D, gamma, xn, D, eps);
        ref_quantize_row_q8_0(xn, xq, D);
        if (dbg_xq)
            memcpy(dbg_xq + (size_t)i * xq_bytes, xq, xq_bytes);
        ref_gemv(qi, wq, xq, bq, QD, D, 0);
        ref_gemv(k, wk, xq, bk, KD, D, 0);
        ref_gemv(v, wv, xq, bv, KD, D, 1);
        ref_rope(qi, k, rope_cos, rope_sin, pos + i, H, KV, hd);
        ref_kv_store(k_cache, v_cache, k, v, pos + i, KV, capacity, hd);
        if (dbg_q)
            memcpy(dbg_q + (size_t)i * QD, qi, sizeof(float) * (size_t)QD);
        if (dbg_k)
            memcpy(dbg_k + (size_t)i * KD, k, sizeof(float) * (size_t)KD);
        if (dbg_v)
            memcpy(dbg_v + (size_t)i * KD, v, sizeof(float) * (size_t)KD);
    }
    /* phase 2: causal attention, then the O projection and the residual */
    for (int i = 0; i < n; ++i) {
        float *oi = out + (size_t)i * D;
        ref_attention(q + (size_t)i * QD, k_cache, v_cache, attn, H, KV, pos + i + 1, capacity, hd);
        if (dbg_attn)
            memcpy(dbg_attn + (size_t)i * QD, attn, sizeof(float) * (size_t)QD);
        ref_quantize_row_q8_0(attn, xq, QD);
        if (dbg_aq)
            memcpy(dbg_aq + (size_t)i * aq_bytes, xq, aq_bytes);
        ref_gemv(oi, wo, xq, bo, D, QD, 0);
        for (int e = 0; e < D; ++e)
            oi[e] = oi[e] + residual[(size_t)i * D + e];
    }
    free(xn);
    free(q);
    free(k);
    free(v);
    free(attn);
    free(xq);
}
