/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for Q8_0 GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or call
 * this file; only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant generator with
 * the CUDA library.
 *
 * What it computes (sources are the pages' titles and sections):
 *
 *  - Q8_0 block quantisation: blocks of 32 values, one fp16 scale per block, int8
 *    codes.  "Engine perf(hip): MTP draft, shared expert, verify/sampler head",
 *    Summary item 4 and "Verification & Parity Evidence" (the warp-per-block
 *    quantize_q8_0_scaled kernel, bitwise equal to a CPU reference on zero, .5-tie
 *    and normal inputs).  The scale rule (max|x| / 127, round to nearest) is the
 *    workload definition of the KV cache.  Readings where the pages are silent:
 *      d32 = amax / 127 in IEEE fp32 division; the stored scale is fp16(d32),
 *      rounded to nearest even; q = clamp(round_half_away_from_zero(x / d32),
 *      -127, 127) with an IEEE fp32 division; a block whose d32 is 0 stores d = 0
 *      and all-zero codes.
 *
 *  - Multi-row causal attention over the dequantised cache (fp64): "perf(gfx1100):
 *    share Q8 KV scans across verifier rows", Summary (one wave owns 4 or 8 query
 *    rows, sequential windows of 4-32 rows) and "Kernel evidence" (dedicated oracle,
 *    worst relative error); "gfx12 WMMA kernel for the int8-KV QSA prompt attention",
 *    "How" and "Measurements" (error vs FP64).  Row i of a call sees keys
 *    [0, q_pos0 + i]; q head h reads kv head h / (Hq / Hkv).
 *      s_n = scale * sum_j q_j * kcode[n][j] * dK[n][j/32]
 *      p_n = exp(s_n - max s) / sum exp(s - max s);  out_j = sum_n p_n vcode[n][j] dV[n][j/32]
 *
 *  - Tree-shaped verify windows (the variant the multi-row route does not admit, "share Q8
 *    KV scans across verifier rows", Summary: sequential windows only).  Reading: the T
 *    window tokens sit at positions q_pos0 .. q_pos0 + T - 1 in the order given; row i sees
 *    every key n < q_pos0 and the window key q_pos0 + j exactly when bit j of mask[i] is
 *    set (j < 32, n < kv_len).  The sequential window is mask[i] = 2^(i+1) - 1.
 *
 *  - fp16 KV pools (the pages' other pool format, which their new kernels leave on the old
 *    path: "gfx12 WMMA kernel for the int8-KV QSA prompt attention", Gating and Limits).
 *    Reading: K and V are stored as IEEE binary16 values, [n_kv_heads][capacity][head_dim];
 *    an append rounds the fp32 inputs to nearest even; attention is the same fp64 formula
 *    with k[n][j] and v[n][j] the stored values (no codes, no block scales).
 *
 *  - K8V4 pools (the pages run a `--kv k8v4` pool and keep it, like fp16, on the older
 *    kernels: "gfx12 WMMA kernel for the int8-KV QSA prompt attention", Gating and Limits;
 *    the 4-bit V format itself is not given).  Reading: K is Q8_0 as above; V is a
 *    symmetric 4-bit block format mirroring the Q8_0 rule with 2^3 - 1 in place of 2^7 - 1:
 *      d32 = amax / 7 (IEEE fp32 division), stored as fp16(d32) rounded to nearest even;
 *      q = clamp(round_half_away_from_zero(x / d32), -7, 7), 0 for a block whose d32 is 0;
 *      stored as the nibble q + 8, element 2m in the low and 2m + 1 in the high nibble of
 *      byte m, [n_kv_heads][capacity][head_dim / 2] bytes; the value is (nibble - 8) * d.
 *
 *  - Split-context partials and their merge ("share Q8 KV scans across verifier
 *    rows", Summary: "The partials layout and reducer are unchanged"): a partial over
 *    keys [k0, k1) is (o, m, l) with m = max s over the visible keys of the range,
 *    l = sum exp(s - m), o = sum exp(s - m) v (unnormalised).  An empty range gives
 *    m = -inf, l = 0, o = 0.  The merge is m* = max m_s, l* = sum l_s exp(m_s - m*),
 *    out = sum o_s exp(m_s - m*) / l*.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QBLOCK 32

/* ---------------------------------------------------------------- fp16 bits */

/* Half-precision bits -> double, from the IEEE 754 binary16 definition:
 * sign s, 5-bit exponent e (bias 15), 10-bit fraction f.
 *   e == 0      : (-1)^s * f * 2^-24            (zero and subnormals)
 *   0 < e < 31  : (-1)^s * (1024 + f) * 2^(e-25)
 *   e == 31     : infinity (f == 0) or NaN       */
double oracle_f16_bits_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return s ? -v : v;
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double n) {
    double fl = floor(n);
    double diff = n - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* fp32 -> fp16 bits, round to nearest, ties to even (IEEE 754 default rounding).
 * The magnitude is expressed as an integer count of the fp16 quantum of its binade,
 * rounded, and re-encoded; the encoding is continuous across binades, so a count
 * that rounds up to the next binade carries into the exponent field by itself. */
uint16_t oracle_f32_to_f16_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    double v = fabs((double)x);
    if (isinf(x) || v >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* 65520 = 65504 + half an ulp: ties go to even = inf */
    if (v < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24, count in [0, 1024] (1024 encodes 2^-14) */
        double n = round_half_even(v * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int e2;
    (void)frexp(v, &e2);          /* v = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                /* v in [2^e, 2^(e+1)), e in [-14, 15] */
    double n = round_half_even(v * ldexp(1.0, 10 - e)); /* count of 2^(e-10), in [1024, 2048] */
    uint32_t bits = (uint32_t)(e + 15) * 1024u + ((uint32_t)n - 1024u);
    return (uint16_t)(sign | bits);
}

/* Array forms of the two conversions above (element by element). */
void oracle_f16_bits_to_f64_array(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_bits_to_f64(h[i]);
}

void oracle_f32_to_f16_bits_array(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16_bits(x[i]);
}

/* ---------------------------------------------------------------- Q8_0 */

/* Quantise one block of 32 fp32 values (see header comment for the rule). */
static void quantize_block(const float* x, int8_t* q, uint16_t* d_bits) {
    float amax = 0.0f;
    for (int j = 0; j < QBLOCK; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float d32 = amax / 127.0f;
    *d_bits = oracle_f32_to_f16_bits(d32);
    for (int j = 0; j < QBLOCK; ++j) {
        if (d32 == 0.0f) {
            q[j] = 0;
            continue;
        }
        float t = x[j] / d32;
        float r = roundf(t); /* C roundf: halfway cases away from zero */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[j] = (int8_t)r;
    }
}

/* Quantise n_blocks consecutive blocks of 32 values. */
void oracle_quantize_q8_0(const float* x, int64_t n_blocks, int8_t* q, uint16_t* d_bits) {
    for (int64_t b = 0; b < n_blocks; ++b)
        quantize_block(x + b * QBLOCK, q + b * QBLOCK, d_bits + b);
}

/* Append n_tok tokens of K (or V) values x[n_tok][n_kv_heads][head_dim] into the
 * plane pair codes[n_kv_heads][capacity][head_dim], scales[n_kv_heads][capacity][head_dim/32]
 * at positions [pos0, pos0 + n_tok).  Returns 0, or -1 on a bad argument. */
int oracle_kv_append_q8_0(const float* x, int n_tok, int n_kv_heads, int head_dim,
                          int8_t* codes, uint16_t* scales, int capacity, int pos0) {
    if (n_tok < 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % QBLOCK) return -1;
    if (pos0 < 0 || (int64_t)pos0 + n_tok > capacity) return -1;
    const int nb = head_dim / QBLOCK;
    for (int t = 0; t < n_tok; ++t)
        for (int h = 0; h < n_kv_heads; ++h) {
            const float* src = x + ((int64_t)t * n_kv_heads + h) * head_dim;
            int64_t row = (int64_t)h * capacity + pos0 + t;
            for (int b = 0; b < nb; ++b)
                quantize_block(src + b * QBLOCK, codes + row * head_dim + b * QBLOCK,
                               scales + row * nb + b);
        }
    return 0;
}

/* ---------------------------------------------------------------- 4-bit V (K8V4) */

/* Quantise one block of 32 fp32 values to 16 bytes of nibbles + an fp16 scale (rule in the
 * header comment). */
static void quantize_block_q4(const float* x, uint8_t* packed, uint16_t* d_bits) {
    float amax = 0.0f;
    for (int j = 0; j < QBLOCK; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float d32 = amax / 7.0f;
    *d_bits = oracle_f32_to_f16_bits(d32);
    for (int m = 0; m < QBLOCK / 2; ++m) packed[m] = 0;
    for (int j = 0; j < QBLOCK; ++j) {
        int q = 0;
        if (d32 != 0.0f) {
            float r = roundf(x[j] / d32);
            if (r > 7.0f) r = 7.0f;
            if (r < -7.0f) r = -7.0f;
            q = (int)r;
        }
        packed[j / 2] |= (uint8_t)((q + 8) << (4 * (j & 1)));
    }
}

void oracle_quantize_q4(const float* x, int64_t n_blocks, uint8_t* packed, uint16_t* d_bits) {
    for (int64_t b = 0; b < n_blocks; ++b)
        quantize_block_q4(x + b * QBLOCK, packed + b * (QBLOCK / 2), d_bits + b);
}

/* Append n_tok tokens of V values x[n_tok][n_kv_heads][head_dim] into the 4-bit plane
 * codes[n_kv_heads][capacity][head_dim/2], scales[n_kv_heads][capacity][head_dim/32] at
 * positions [pos0, pos0 + n_tok).  Returns 0, or -1 on a bad argument. */
int oracle_kv_append_q4(const float* x, int n_tok, int n_kv_heads, int head_dim, uint8_t* codes,
                        uint16_t* scales, int capacity, int pos0) {
    if (n_tok < 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % QBLOCK) return -1;
    if (pos0 < 0 || (int64_t)pos0 + n_tok > capacity) return -1;
    const int nb = head_dim / QBLOCK;
    for (int t = 0; t < n_tok; ++t)
        for (int h = 0; h < n_kv_heads; ++h) {
            const float* src = x + ((int64_t)t * n_kv_heads + h) * head_dim;
            int64_t row = (int64_t)h * capacity + pos0 + t;
            for (int b = 0; b < nb; ++b)
                quantize_block_q4(src + b * QBLOCK, codes + row * (head_dim / 2) + b * (QBLOCK / 2),
                                  scales + row * nb + b);
        }
    return 0;
}

/* ---------------------------------------------------------------- attention */

typedef struct {
    const int8_t* k_codes;
    const uint16_t* k_scales;
    const int8_t* v_codes;
    const uint16_t* v_scales;
    int n_kv_heads, head_dim, capacity;
    int format;              /* ORACLE_Q8_0, ORACLE_F16 or ORACLE_K8V4 */
    const uint16_t* k_f16;   /* ORACLE_F16: fp16 bits [n_kv_heads][capacity][head_dim] */
    const uint16_t* v_f16;
    const uint8_t* v_q4;     /* ORACLE_K8V4: V nibbles [n_kv_heads][capacity][head_dim/2] (scales in v_scales) */
} oracle_cache;

enum { ORACLE_Q8_0 = 0, ORACLE_F16 = 1, ORACLE_K8V4 = 2 };

/* Value of element j of token n of kv head h in one plane: code * block scale for Q8_0,
 * the stored binary16 value for an fp16 pool. */
static double deq_plane(const oracle_cache* c, int plane, int h, int64_t n, int j) {
    int64_t row = (int64_t)h * c->capacity + n;
    if (c->format == ORACLE_F16)
        return oracle_f16_bits_to_f64((plane ? c->v_f16 : c->k_f16)[row * c->head_dim + j]);
    if (c->format == ORACLE_K8V4 && plane) {
        uint8_t byte = c->v_q4[row * (c->head_dim / 2) + j / 2];
        int nib = (j & 1) ? (byte >> 4) : (byte & 15);
        double d = oracle_f16_bits_to_f64(c->v_scales[row * (c->head_dim / QBLOCK) + j / QBLOCK]);
        return (double)(nib - 8) * d;
    }
    const int8_t* codes = plane ? c->v_codes : c->k_codes;
    const uint16_t* scales = plane ? c->v_scales : c->k_scales;
    double d = oracle_f16_bits_to_f64(scales[row * (c->head_dim / QBLOCK) + j / QBLOCK]);
    return (double)codes[row * c->head_dim + j] * d;
}
#define deq_k(c, h, n, j) deq_plane((c), 0, (h), (n), (j))
#define deq_v(c, h, n, j) deq_plane((c), 1, (h), (n), (j))

/* Append n_tok fp32 tokens [n_tok][n_kv_heads][head_dim] to an fp16 plane at pos0 (round to
 * nearest even).  Returns 0, or -1 for bad arguments. */
int oracle_kv_append_f16(const float* x, int n_tok, int n_kv_heads, int head_dim, uint16_t* plane,
                         int capacity, int pos0) {
    if (!x || !plane || n_tok < 0 || n_kv_heads <= 0 || head_dim <= 0 || pos0 < 0 ||
        (int64_t)pos0 + n_tok > capacity)
        return -1;
    for (int t = 0; t < n_tok; ++t)
        for (int h = 0; h < n_kv_heads; ++h)
            for (int j = 0; j < head_dim; ++j)
                plane[((int64_t)h * capacity + pos0 + t) * head_dim + j] =
                    oracle_f32_to_f16_bits(x[((int64_t)t * n_kv_heads + h) * head_dim + j]);
    return 0;
}

/* One (query row, q head): softmax attention over keys [k0, min(k1, q_pos0+i+1)).
 * Writes the unnormalised partial (o, m, l) for that key range. */
static void attend_one(const oracle_cache* c, const double* qrow, int kv_head, int64_t k0, int64_t k1,
                       double scale, double* o, double* m_out, double* l_out, double* s_buf) {
    const int hd = c->head_dim;
    for (int j = 0; j < hd; ++j) o[j] = 0.0;
    if (k1 <= k0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int64_t n = k0; n < k1; ++n) {
        double s = 0.0;
        for (int j = 0; j < hd; ++j) s += qrow[j] * deq_k(c, kv_head, n, j);
        s *= scale;
        s_buf[n - k0] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int64_t n = k0; n < k1; ++n) {
        double p = exp(s_buf[n - k0] - m);
        l += p;
        for (int j = 0; j < hd; ++j) o[j] += p * deq_v(c, kv_head, n, j);
    }
    *m_out = m;
    *l_out = l;
}

static int check_cache(const oracle_cache* c, int n_q_heads, int kv_len) {
    if (!c || c->n_kv_heads <= 0 || c->head_dim <= 0 || c->head_dim % QBLOCK) return -1;
    if (c->format != ORACLE_Q8_0 && c->format != ORACLE_F16 && c->format != ORACLE_K8V4) return -1;
    if (n_q_heads <= 0 || n_q_heads % c->n_kv_heads) return -1;
    if (kv_len < 0 || kv_len > c->capacity) return -1;
    return 0;
}

/* Attention partials over keys [key_begin, key_end) for selected (row, head) pairs.
 *   q        : fp64 [n_q][n_q_heads][head_dim]
 *   sel_row, sel_head : n_sel pairs (row i in [0, n_q), q head h); if sel_row is NULL,
 *              every (i, h) in row-major order is computed (n_sel must be n_q * n_q_heads)
 *   o        : fp64 [n_sel][head_dim], m, l : fp64 [n_sel]
 * Row i sees keys n <= q_pos0 + i and n < kv_len.  Returns 0 or -1. */
int oracle_attention_partial(const oracle_cache* c, const double* q, int n_q, int n_q_heads,
                             int kv_len, int q_pos0, double scale, int64_t key_begin, int64_t key_end,
                             const int32_t* sel_row, const int32_t* sel_head, int64_t n_sel,
                             double* o, double* m, double* l) {
    if (check_cache(c, n_q_heads, kv_len) || n_q < 0 || q_pos0 < 0) return -1;
    if (!sel_row && n_sel != (int64_t)n_q * n_q_heads) return -1;
    const int g = n_q_heads / c->n_kv_heads;
    const int hd = c->head_dim;
    int bad = 0;
#pragma omp parallel
    {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n_sel; ++t) {
            int i = sel_row ? sel_row[t] : (int)(t / n_q_heads);
            int h = sel_row ? sel_head[t] : (int)(t % n_q_heads);
            if (i < 0 || i >= n_q || h < 0 || h >= n_q_heads || !s_buf) {
                bad = 1;
                continue;
            }
            int64_t vis_end = (int64_t)q_pos0 + i + 1;
            if (vis_end > kv_len) vis_end = kv_len;
            int64_t k0 = key_begin < 0 ? 0 : key_begin;
            int64_t k1 = key_end < vis_end ? key_end : vis_end;
            attend_one(c, q + ((int64_t)i * n_q_heads + h) * hd, h / g, k0, k1, scale,
                       o + t * hd, m + t, l + t, s_buf);
        }
        free(s_buf);
    }
    return bad ? -1 : 0;
}

/* Normalised attention output for selected (row, head) pairs: out = o / l over all visible keys. */
int oracle_attention(const oracle_cache* c, const double* q, int n_q, int n_q_heads, int kv_len,
                     int q_pos0, double scale, const int32_t* sel_row, const int32_t* sel_head,
                     int64_t n_sel, double* out) {
    double* m = (double*)malloc(sizeof(double) * (size_t)(n_sel > 0 ? n_sel : 1));
    double* l = (double*)malloc(sizeof(double) * (size_t)(n_sel > 0 ? n_sel : 1));
    if (!m || !l) { free(m); free(l); return -1; }
    int rc = oracle_attention_partial(c, q, n_q, n_q_heads, kv_len, q_pos0, scale, 0, kv_len,
                                      sel_row, sel_head, n_sel, out, m, l);
    if (rc == 0) {
        const int hd = c->head_dim;
        for (int64_t t = 0; t < n_sel; ++t)
            for (int j = 0; j < hd; ++j) out[t * hd + j] = (l[t] > 0.0) ? out[t * hd + j] / l[t] : 0.0;
    }
    free(m);
    free(l);
    return rc;
}

/* One (query row, q head): softmax attention over an explicit ascending list of keys. */
static void attend_list(const oracle_cache* c, const double* qrow, int kv_head, const int64_t* keys, int64_t n_keys,
                        double scale, double* out, double* s_buf) {
    const int hd = c->head_dim;
    for (int j = 0; j < hd; ++j) out[j] = 0.0;
    if (n_keys <= 0) return;
    double m = -INFINITY;
    for (int64_t t = 0; t < n_keys; ++t) {
        double s = 0.0;
        for (int j = 0; j < hd; ++j) s += qrow[j] * deq_k(c, kv_head, keys[t], j);
        s *= scale;
        s_buf[t] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) {
        double p = exp(s_buf[t] - m);
        l += p;
        for (int j = 0; j < hd; ++j) out[j] += p * deq_v(c, kv_head, keys[t], j);
    }
    for (int j = 0; j < hd; ++j) out[j] /= l;
}

/* Normalised attention of a tree-shaped window for selected (row, head) pairs: row i sees
 * the keys n < min(q_pos0, kv_len) and q_pos0 + j (< kv_len) for every bit j of mask[i].
 * A row with no visible key gives zeros.  Returns 0 or -1. */
int oracle_attention_tree(const oracle_cache* c, const double* q, int n_q, int n_q_heads, int kv_len,
                          int q_pos0, const uint32_t* mask, double scale, const int32_t* sel_row,
                          const int32_t* sel_head, int64_t n_sel, double* out) {
    if (check_cache(c, n_q_heads, kv_len) || n_q < 0 || n_q > 32 || q_pos0 < 0 || !mask) return -1;
    if (!sel_row && n_sel != (int64_t)n_q * n_q_heads) return -1;
    const int g = n_q_heads / c->n_kv_heads;
    const int hd = c->head_dim;
    int bad = 0;
#pragma omp parallel
    {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(kv_len > 0 ? kv_len : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n_sel; ++t) {
            int i = sel_row ? sel_row[t] : (int)(t / n_q_heads);
            int h = sel_row ? sel_head[t] : (int)(t % n_q_heads);
            if (i < 0 || i >= n_q || h < 0 || h >= n_q_heads || !s_buf || !keys) {
                bad = 1;
                continue;
            }
            int64_t n_keys = 0;
            for (int64_t n = 0; n < q_pos0 && n < kv_len; ++n) keys[n_keys++] = n;
            for (int j = 0; j < 32; ++j)
                if (((mask[i] >> j) & 1u) && (int64_t)q_pos0 + j < kv_len) keys[n_keys++] = (int64_t)q_pos0 + j;
            attend_list(c, q + ((int64_t)i * n_q_heads + h) * hd, h / g, keys, n_keys, scale, out + t * hd, s_buf);
        }
        free(s_buf);
        free(keys);
    }
    return bad ? -1 : 0;
}

/* Merge n_split partials: part_o [n_split][rows][hd], part_m / part_l [n_split][rows]
 * -> out [rows][hd].  A row whose every partial is empty (m = -inf) gives zeros. */
int oracle_combine(const double* part_o, const double* part_m, const double* part_l, int n_split,
                   int64_t rows, int hd, double* out) {
    if (n_split <= 0 || rows < 0 || hd <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double ms = -INFINITY;
        for (int s = 0; s < n_split; ++s)
            if (part_m[(int64_t)s * rows + r] > ms) ms = part_m[(int64_t)s * rows + r];
        double* dst = out + r * hd;
        for (int j = 0; j < hd; ++j) dst[j] = 0.0;
        if (ms == -INFINITY) continue;
        double ls = 0.0;
        for (int s = 0; s < n_split; ++s) {
            double w = exp(part_m[(int64_t)s * rows + r] - ms);
            ls += part_l[(int64_t)s * rows + r] * w;
            const double* src = part_o + ((int64_t)s * rows + r) * hd;
            for (int j = 0; j < hd; ++j) dst[j] += src[j] * w;
        }
        for (int j = 0; j < hd; ++j) dst[j] /= ls;
    }
    return 0;
}

/* ---------------------------------------------------------------- threads */

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
