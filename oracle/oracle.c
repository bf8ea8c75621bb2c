/*
 * Reference ("oracle") implementation of the block-quantized weight matmul
 *
 *     y[m, n] = sum_k dequant(W)[n, k] * x[m, k]
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls this file: only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg do. It shares no code, header, table or
 * helper with the CUDA library; the two are written separately from the same block-format specification,
 * whose layouts, decoding rule and encoder are restated in the functions below.
 *
 * What it computes, and where that comes from:
 *   - The method: each weight block is dequantized and then multiplied by the activation rows (candle
 *     PR 4056, "Metal: 64-token tile for the quantized matrix-matrix kernel", section "Why the tile sets
 *     the weight reuse": the threadgroup reads the quantized blocks, dequantizes them and multiplies them
 *     by the tokens). Because the tiling only changes how often a weight is re-read, the result the
 *     method reaches is the plain definition above, which is what this file writes out.
 *   - The expert-indexed product y[t, j, :] = W_{ids[t, j]} x[t, :] (llama.cpp PR 28086, "metal : fix
 *     idle threads in mul_mv_iq3_xxs for ne00 < 1024", sections "Overview" and "Additional
 *     information": MUL_MAT_ID, one mat-vec per routed expert), and its form with one activation row per
 *     (token, slot), y[t, j, :] = W_{ids[t, j]} x[t, j, :] (the same page, "Test methodology": the
 *     experts' down projection, ffn_down_exps, whose input differs per routed expert).
 *   - The block layouts, the exact decoding rule and the deterministic encoder: the pages name the types
 *     (candle PR 4056, section "What changes"; tiny-llm PR 122, "Summary") but define none of them, so
 *     they follow this repository's block-format specification, sections 2 to 4.
 *
 * Precision: decoding is exact in binary64 (every field value and every product in the formulas is
 * exact there); the dot product is a plain ascending-k binary64 loop. The encoder takes its rounding
 * decisions in binary32, as the specification fixes, so that an independent device encoder can agree
 * with it bit for bit. Build with -ffp-contract=off and without fast-math.
 *
 * Parity pins: every function here is pinned by tests in tests/test_oracle*.py against facts that do not
 * come from this file (numpy/torch conversions, hand-built blocks, exact rational dot products,
 * permutation invariance, round-trip bounds).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    T_F32 = 0, T_F16 = 1, T_BF16 = 2, T_Q4_0 = 3, T_Q4_1 = 4, T_Q5_0 = 5, T_Q5_1 = 6, T_Q8_0 = 7,
    T_Q2_K = 8, T_Q3_K = 9, T_Q4_K = 10, T_Q5_K = 11, T_Q6_K = 12, T_A4G64 = 13, T_COUNT = 14
};

/* Block size (weights) and bytes per block, specification section 1. */
static const int QK[T_COUNT] = {1, 1, 1, 32, 32, 32, 32, 32, 256, 256, 256, 256, 256, 64};
static const int QB[T_COUNT] = {4, 2, 2, 18, 20, 22, 24, 34, 84, 110, 144, 176, 210, 36};

int orc_type_info(int qt, int *qk, int *bytes)
{
    if (qt < 0 || qt >= T_COUNT) return -1;
    *qk = QK[qt];
    *bytes = QB[qt];
    return 0;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- half-precision codecs */

/* IEEE binary16 -> exact binary64. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);    /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> exact binary64: the value of the binary32 whose upper half it is. */
double orc_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 255;
    int f = h & 127;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);              /* subnormal: f * 2^-133 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);    /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/*
 * Round a binary32 to a format with `p` significand bits (hidden bit included) and minimum normal
 * exponent `emin`, to nearest, ties to even. Returns the magnitude's bit pattern: the quantum at binade
 * E (clamped to emin for subnormals) is 2^(E - p + 1); the rounded value is r quanta, and the pattern is
 * (E - emin) * 2^(p-1) + r. A carry out of the significand (r = 2^p) lands on the next binade's pattern
 * by the same formula, and past the top binade on the infinity pattern.
 */
static uint32_t round_to_format(double a, int p, int emin)
{
    if (a == 0.0) return 0;
    int e2;
    frexp(a, &e2);               /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;              /* a in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;
    double r = nearbyint(ldexp(a, -(E - p + 1)));   /* exact scaling, then round half to even */
    return (uint32_t)(E - emin) * (1u << (p - 1)) + (uint32_t)r;
}

/* binary32 -> IEEE binary16, round to nearest even (specification section 4, f16()). */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)f);
    if (isinf(f) || a >= 65520.0) return (uint16_t)(sign | 0x7C00u);  /* 65520 is the tie above 65504 */
    return (uint16_t)(sign | round_to_format(a, 11, -14));
}

/* binary32 -> bfloat16, round to nearest even (specification section 4, bf16()). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(f)) return (uint16_t)(sign | 0x7F80u);
    uint32_t m = round_to_format(fabs((double)f), 8, -126);
    if (m > 0x7F80u) m = 0x7F80u;
    return (uint16_t)(sign | m);
}

static float f16f(uint16_t h) { return (float)orc_f16_to_f64(h); }
static float bf16f(uint16_t h) { return (float)orc_bf16_to_f64(h); }

/* ---------------------------------------------------------------- byte-field readers */

static unsigned rd8(const uint8_t *b, int off) { return b[off]; }
static unsigned rd16(const uint8_t *b, int off) { return (unsigned)b[off] | ((unsigned)b[off + 1] << 8); }

/* Bit `pos` .. pos+width-1 of the little-endian integer formed by the bytes starting at b[off]. */
static unsigned rdbits(const uint8_t *b, int off, int pos, int width)
{
    unsigned v = 0;
    for (int t = 0; t < width; t++) {
        int p = pos + t;
        v |= (unsigned)((b[off + p / 8] >> (p % 8)) & 1) << t;
    }
    return v;
}

static void wr16(uint8_t *b, int off, unsigned v) { b[off] = (uint8_t)(v & 255); b[off + 1] = (uint8_t)(v >> 8); }

static void wrbits(uint8_t *b, int off, int pos, int width, unsigned v)
{
    for (int t = 0; t < width; t++) {
        int p = pos + t;
        uint8_t bit = (uint8_t)(1u << (p % 8));
        if ((v >> t) & 1) b[off + p / 8] |= bit;
        else b[off + p / 8] &= (uint8_t)~bit;
    }
}

/* ---------------------------------------------------------------- element code readers (spec. section 2) */

/* nibble order N32: 16 bytes at `off` hold 32 codes. */
static unsigned nib32(const uint8_t *b, int off, int i) { return i < 16 ? (b[off + i] & 15) : (b[off + i - 16] >> 4); }
/* bit plane P32: bit i of the 32-bit little-endian word at `off`. */
static unsigned bit32(const uint8_t *b, int off, int i) { return (b[off + i / 8] >> (i % 8)) & 1; }
/* Q2_K / Q3_K two-bit codes: 64 bytes at `off`. */
static unsigned two256(const uint8_t *b, int off, int i)
{
    int h = i / 128, g = (i % 128) / 32, l = i % 32;
    return (b[off + 32 * h + l] >> (2 * g)) & 3;
}
/* Q4_K / Q5_K four-bit codes: 128 bytes at `off`. */
static unsigned nib256(const uint8_t *b, int off, int i)
{
    int c = i / 64, l = i % 32;
    unsigned v = b[off + 32 * c + l];
    return (i % 64) < 32 ? (v & 15) : (v >> 4);
}

/* ---------------------------------------------------------------- decoding (spec. section 3) */

/*
 * Decode one block of type qt to exact binary64 values. Every field is read as its exact value and the
 * formula of section 1 is evaluated in binary64, where it is exact.
 */
static void decode_block(int qt, const uint8_t *b, double *w)
{
    switch (qt) {
    case T_F32: { float v; memcpy(&v, b, 4); w[0] = (double)v; break; }
    case T_F16: w[0] = orc_f16_to_f64((uint16_t)rd16(b, 0)); break;
    case T_BF16: w[0] = orc_bf16_to_f64((uint16_t)rd16(b, 0)); break;
    case T_Q4_0: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 0));
        for (int i = 0; i < 32; i++) w[i] = d * ((double)nib32(b, 2, i) - 8.0);
        break;
    }
    case T_Q4_1: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 0)), m = orc_f16_to_f64((uint16_t)rd16(b, 2));
        for (int i = 0; i < 32; i++) w[i] = d * (double)nib32(b, 4, i) + m;
        break;
    }
    case T_Q5_0: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 0));
        for (int i = 0; i < 32; i++) w[i] = d * ((double)(nib32(b, 6, i) + 16 * bit32(b, 2, i)) - 16.0);
        break;
    }
    case T_Q5_1: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 0)), m = orc_f16_to_f64((uint16_t)rd16(b, 2));
        for (int i = 0; i < 32; i++) w[i] = d * (double)(nib32(b, 8, i) + 16 * bit32(b, 4, i)) + m;
        break;
    }
    case T_Q8_0: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 0));
        for (int i = 0; i < 32; i++) w[i] = d * (double)(int8_t)b[2 + i];
        break;
    }
    case T_Q2_K: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 80)), dmin = orc_f16_to_f64((uint16_t)rd16(b, 82));
        for (int i = 0; i < 256; i++) {
            unsigned sm = rd8(b, i / 16);
            w[i] = d * (double)(sm & 15) * (double)two256(b, 16, i) - dmin * (double)(sm >> 4);
        }
        break;
    }
    case T_Q3_K: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 108));
        for (int i = 0; i < 256; i++) {
            int sc = (int)rdbits(b, 96, 6 * (i / 16), 6) - 32;
            int q = (int)(two256(b, 32, i) + 4 * ((b[i % 32] >> (i / 32)) & 1)) - 4;
            w[i] = d * (double)sc * (double)q;
        }
        break;
    }
    case T_Q4_K:
    case T_Q5_K: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 0)), dmin = orc_f16_to_f64((uint16_t)rd16(b, 2));
        for (int i = 0; i < 256; i++) {
            int s = i / 32;
            unsigned sc = rdbits(b, 4, 6 * s, 6), mn = rdbits(b, 4, 48 + 6 * s, 6);
            unsigned q = (qt == T_Q4_K) ? nib256(b, 16, i)
                                        : nib256(b, 48, i) + 16 * ((b[16 + i % 32] >> (i / 32)) & 1);
            w[i] = d * (double)sc * (double)q - dmin * (double)mn;
        }
        break;
    }
    case T_Q6_K: {
        double d = orc_f16_to_f64((uint16_t)rd16(b, 208));
        for (int i = 0; i < 256; i++) {
            int h = i / 128, j = i % 128;
            unsigned lo = (b[64 * h + j % 64] >> (4 * (j / 64))) & 15;
            unsigned hi = (b[128 + 32 * h + j % 32] >> (2 * (j / 32))) & 3;
            int sc = (int8_t)b[192 + i / 16];
            w[i] = d * (double)sc * ((double)(lo + 16 * hi) - 32.0);
        }
        break;
    }
    case T_A4G64: {
        double s = orc_bf16_to_f64((uint16_t)rd16(b, 0)), bb = orc_bf16_to_f64((uint16_t)rd16(b, 2));
        for (int i = 0; i < 64; i++) {
            unsigned q = i < 32 ? (b[4 + i] & 15) : (b[4 + i - 32] >> 4);
            w[i] = s * (double)q + bb;
        }
        break;
    }
    }
}

/* Dequantize an N x K matrix to exact binary64 values (row-major out[n*K + k]). */
int orc_dequant_f64(int qt, const uint8_t *wq, int64_t N, int64_t K, double *out)
{
    if (qt < 0 || qt >= T_COUNT || K % QK[qt] != 0) return -1;
    int64_t nb = K / QK[qt];
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            decode_block(qt, wq + (n * nb + b) * QB[qt], out + n * K + b * QK[qt]);
    return 0;
}

/* The same values rounded once to binary32 (the rule a device decoder must meet, spec. section 3). */
int orc_dequant_f32(int qt, const uint8_t *wq, int64_t N, int64_t K, float *out)
{
    if (qt < 0 || qt >= T_COUNT || K % QK[qt] != 0) return -1;
    int64_t nb = K / QK[qt];
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
        double tmp[256];
        for (int64_t b = 0; b < nb; b++) {
            decode_block(qt, wq + (n * nb + b) * QB[qt], tmp);
            for (int i = 0; i < QK[qt]; i++) {
                if (qt == T_F32) {       /* keep the stored bits, NaN payloads included */
                    memcpy(&out[n * K + b * QK[qt] + i], wq + (n * nb + b) * 4, 4);
                } else {
                    out[n * K + b * QK[qt] + i] = (float)tmp[i];
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- encoding (spec. section 4) */

static float clampf(float t, float a, float b) { return t < a ? a : (t > b ? b : t); }
static int rne_clamp(float t, float a, float b) { return (int)rintf(clampf(t, a, b)); }

static void group_stats(const float *w, int n, float *amax, float *lo, float *hi)
{
    float am = 0.0f, l = w[0], h = w[0];
    for (int i = 0; i < n; i++) {
        float a = fabsf(w[i]);
        if (a > am) am = a;
        if (w[i] < l) l = w[i];
        if (w[i] > h) h = w[i];
    }
    *amax = am; *lo = l; *hi = h;
}

static void put_nib32(uint8_t *b, int off, int i, unsigned q)
{
    if (i < 16) b[off + i] = (uint8_t)((b[off + i] & 0xF0) | q);
    else b[off + i - 16] = (uint8_t)((b[off + i - 16] & 0x0F) | (q << 4));
}

static void encode_block(int qt, const float *w, uint8_t *b)
{
    memset(b, 0, (size_t)QB[qt]);
    switch (qt) {
    case T_F32: memcpy(b, w, 4); break;
    case T_F16: wr16(b, 0, orc_f32_to_f16(w[0])); break;
    case T_BF16: wr16(b, 0, orc_f32_to_bf16(w[0])); break;
    case T_Q4_0:
    case T_Q5_0:
    case T_Q8_0: {
        float amax, lo, hi;
        group_stats(w, 32, &amax, &lo, &hi);
        float top = qt == T_Q4_0 ? 7.0f : (qt == T_Q5_0 ? 15.0f : 127.0f);
        float bot = qt == T_Q4_0 ? -8.0f : (qt == T_Q5_0 ? -16.0f : -127.0f);
        uint16_t dh = orc_f32_to_f16(amax / top);
        float D = f16f(dh);
        wr16(b, 0, dh);
        for (int i = 0; i < 32; i++) {
            int q = D == 0.0f ? 0 : rne_clamp(w[i] / D, bot, top);
            if (qt == T_Q4_0) put_nib32(b, 2, i, (unsigned)(q + 8));
            else if (qt == T_Q5_0) {
                unsigned u = (unsigned)(q + 16);
                put_nib32(b, 6, i, u & 15);
                if (u >> 4) b[2 + i / 8] |= (uint8_t)(1u << (i % 8));
            } else b[2 + i] = (uint8_t)(int8_t)q;
        }
        break;
    }
    case T_Q4_1:
    case T_Q5_1: {
        float amax, lo, hi;
        group_stats(w, 32, &amax, &lo, &hi);
        float top = qt == T_Q4_1 ? 15.0f : 31.0f;
        uint16_t dh = orc_f32_to_f16((hi - lo) / top), mh = orc_f32_to_f16(lo);
        float D = f16f(dh), Mv = f16f(mh);
        wr16(b, 0, dh);
        wr16(b, 2, mh);
        for (int i = 0; i < 32; i++) {
            int q = D == 0.0f ? 0 : rne_clamp((w[i] - Mv) / D, 0.0f, top);
            if (qt == T_Q4_1) put_nib32(b, 4, i, (unsigned)q);
            else {
                put_nib32(b, 8, i, (unsigned)q & 15);
                if (q >> 4) b[4 + i / 8] |= (uint8_t)(1u << (i % 8));
            }
        }
        break;
    }
    case T_A4G64: {
        float amax, lo, hi;
        group_stats(w, 64, &amax, &lo, &hi);
        uint16_t sh = orc_f32_to_bf16((hi - lo) / 15.0f), bh = orc_f32_to_bf16(lo);
        float S = bf16f(sh), B = bf16f(bh);
        wr16(b, 0, sh);
        wr16(b, 2, bh);
        for (int i = 0; i < 64; i++) {
            unsigned q = S == 0.0f ? 0u : (unsigned)rne_clamp((w[i] - B) / S, 0.0f, 15.0f);
            if (i < 32) b[4 + i] = (uint8_t)((b[4 + i] & 0xF0) | q);
            else b[4 + i - 32] = (uint8_t)((b[4 + i - 32] & 0x0F) | (q << 4));
        }
        break;
    }
    case T_Q2_K:
    case T_Q4_K:
    case T_Q5_K: {
        /* affine K-quants: sub-blocks of 16 (Q2_K) or 32 (Q4_K, Q5_K) */
        int sub = qt == T_Q2_K ? 16 : 32, ns = 256 / sub;
        float levels = qt == T_Q2_K ? 3.0f : (qt == T_Q4_K ? 15.0f : 31.0f);
        float smax = qt == T_Q2_K ? 15.0f : 63.0f;
        float r[16], nn[16], rmax = 0.0f, nmax = 0.0f;
        for (int s = 0; s < ns; s++) {
            float amax, lo, hi;
            group_stats(w + s * sub, sub, &amax, &lo, &hi);
            float l = lo < 0.0f ? lo : 0.0f;
            r[s] = (hi - l) / levels;
            nn[s] = -l;
            if (r[s] > rmax) rmax = r[s];
            if (nn[s] > nmax) nmax = nn[s];
        }
        uint16_t dh = orc_f32_to_f16(rmax / smax), mh = orc_f32_to_f16(nmax / smax);
        float D = f16f(dh), Dm = f16f(mh);
        int doff = qt == T_Q2_K ? 80 : 0;
        wr16(b, doff, dh);
        wr16(b, doff + 2, mh);
        for (int s = 0; s < ns; s++) {
            int sc = D == 0.0f ? 0 : rne_clamp(r[s] / D, 0.0f, smax);
            int mn = Dm == 0.0f ? 0 : rne_clamp(nn[s] / Dm, 0.0f, smax);
            if (qt == T_Q2_K) b[s] = (uint8_t)(sc | (mn << 4));
            else {
                wrbits(b, 4, 6 * s, 6, (unsigned)sc);
                wrbits(b, 4, 48 + 6 * s, 6, (unsigned)mn);
            }
            float S = D * (float)sc, Bm = Dm * (float)mn;   /* exact in binary32 */
            for (int t = 0; t < sub; t++) {
                int i = s * sub + t;
                unsigned q = S == 0.0f ? 0u : (unsigned)rne_clamp((w[i] + Bm) / S, 0.0f, levels);
                if (qt == T_Q2_K) {
                    int h = i / 128, g = (i % 128) / 32, l = i % 32;
                    b[16 + 32 * h + l] |= (uint8_t)(q << (2 * g));
                } else {
                    int c = i / 64, l = i % 32, qoff = qt == T_Q4_K ? 16 : 48;
                    if ((i % 64) < 32) b[qoff + 32 * c + l] |= (uint8_t)(q & 15);
                    else b[qoff + 32 * c + l] |= (uint8_t)((q & 15) << 4);
                    if (qt == T_Q5_K && (q >> 4)) b[16 + i % 32] |= (uint8_t)(1u << (i / 32));
                }
            }
        }
        break;
    }
    case T_Q3_K:
    case T_Q6_K: {
        /* symmetric K-quants, sub-blocks of 16 */
        float top = qt == T_Q3_K ? 3.0f : 31.0f, smax = qt == T_Q3_K ? 31.0f : 127.0f;
        float bot = qt == T_Q3_K ? -4.0f : -32.0f;
        float r[16], rmax = 0.0f;
        for (int s = 0; s < 16; s++) {
            float amax, lo, hi;
            group_stats(w + 16 * s, 16, &amax, &lo, &hi);
            r[s] = amax / top;
            if (r[s] > rmax) rmax = r[s];
        }
        uint16_t dh = orc_f32_to_f16(rmax / smax);
        float D = f16f(dh);
        wr16(b, qt == T_Q3_K ? 108 : 208, dh);
        for (int s = 0; s < 16; s++) {
            int sc = D == 0.0f ? 0 : rne_clamp(r[s] / D, 0.0f, smax);
            if (qt == T_Q3_K) wrbits(b, 96, 6 * s, 6, (unsigned)(sc + 32));
            else b[192 + s] = (uint8_t)(int8_t)sc;
            float S = D * (float)sc;
            for (int t = 0; t < 16; t++) {
                int i = 16 * s + t;
                int q = S == 0.0f ? 0 : rne_clamp(w[i] / S, bot, top);
                if (qt == T_Q3_K) {
                    unsigned u = (unsigned)(q + 4);
                    int h = i / 128, g = (i % 128) / 32, l = i % 32;
                    b[32 + 32 * h + l] |= (uint8_t)((u & 3) << (2 * g));
                    if (u >> 2) b[i % 32] |= (uint8_t)(1u << (i / 32));
                } else {
                    unsigned u = (unsigned)(q + 32);
                    int h = i / 128, j = i % 128;
                    b[64 * h + j % 64] |= (uint8_t)((u & 15) << (4 * (j / 64)));
                    b[128 + 32 * h + j % 32] |= (uint8_t)((u >> 4) << (2 * (j / 32)));
                }
            }
        }
        break;
    }
    }
}

/* Quantize an N x K binary32 matrix into blocks (spec. section 4). */
int orc_quantize(int qt, const float *w, int64_t N, int64_t K, uint8_t *out)
{
    if (qt < 0 || qt >= T_COUNT || K % QK[qt] != 0) return -1;
    int64_t nb = K / QK[qt];
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            encode_block(qt, w + n * K + b * QK[qt], out + (n * nb + b) * QB[qt]);
    return 0;
}

/* ---------------------------------------------------------------- the product */

static double x_at(const void *x, int xbf16, int64_t idx)
{
    if (xbf16) return orc_bf16_to_f64(((const uint16_t *)x)[idx]);
    return (double)((const float *)x)[idx];
}

/*
 * The product on decoded weights: y64[m*N + n] = sum_k w[n,k] x[m,k], k ascending, binary64;
 * bound[m*N + n] = sum_k |w[n,k] x[m,k]|. w is an N x K binary64 matrix. Either output may be NULL.
 */
int orc_matmul_f64(const double *w, int64_t N, int64_t K, int xbf16, const void *x, int64_t M, double *y64,
                   double *bound)
{
    double *xd = (double *)malloc((size_t)(M * K) * sizeof(double));
    if (!xd) return -2;
    for (int64_t i = 0; i < M * K; i++) xd[i] = x_at(x, xbf16, i);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < N; n++) {
        for (int64_t m = 0; m < M; m++) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = w[n * K + k] * xd[m * K + k];
                s += p;
                a += fabs(p);
            }
            if (y64) y64[m * N + n] = s;
            if (bound) bound[m * N + n] = a;
        }
    }
    free(xd);
    return 0;
}

/* The whole method: decode every block exactly (orc_dequant_f64), then the product above. */
int orc_qmm(int qt, int xbf16, const uint8_t *wq, int64_t N, int64_t K, const void *x, int64_t M,
            double *y64, double *bound)
{
    if (qt < 0 || qt >= T_COUNT || K % QK[qt] != 0) return -1;
    double *w = (double *)malloc((size_t)(N * K) * sizeof(double));
    if (!w) return -2;
    orc_dequant_f64(qt, wq, N, K, w);
    int rc = orc_matmul_f64(w, N, K, xbf16, x, M, y64, bound);
    free(w);
    return rc;
}

/* The same sums for a list of (m, n) pairs only: decode just the rows asked for. */
int orc_qmm_sampled(int qt, int xbf16, const uint8_t *wq, int64_t N, int64_t K, const void *x, int64_t M,
                    int64_t npairs, const int64_t *ms, const int64_t *ns, double *y64, double *bound)
{
    if (qt < 0 || qt >= T_COUNT || K % QK[qt] != 0) return -1;
    int64_t nb = K / QK[qt];
    int64_t rowbytes = nb * QB[qt];
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < npairs; p++) {
        int64_t m = ms[p], n = ns[p];
        if (m < 0 || m >= M || n < 0 || n >= N) { bad = 1; continue; }
        double *w = (double *)malloc((size_t)K * sizeof(double));
        orc_dequant_f64(qt, wq + n * rowbytes, 1, K, w);
        double s = 0.0, a = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double pr = w[k] * x_at(x, xbf16, m * K + k);
            s += pr;
            a += fabs(pr);
        }
        y64[p] = s;
        bound[p] = a;
        free(w);
    }
    return bad ? -3 : 0;
}

/*
 * Expert-indexed product: y64[(t*topk + j)*N + n] = sum_k W_e[n,k] x[r,k] with e = ids[t*topk + j], where
 * the activation row r is the token's, r = t (one row per token, shared by its topk slots), or the slot's
 * own, r = t*topk + j (x_per_slot: each routed pair has its own input row, as the down projection of the
 * experts has; llama.cpp PR 28086, "Test methodology", ffn_down_exps).
 * wq[e] points at expert e's N x K block matrix. An id outside [0, E) gives NaN for that slot.
 */
static int qmm_id_rows(int qt, int xbf16, const uint8_t *const *wq, int64_t E, int64_t N, int64_t K,
                       const void *x, int x_per_slot, const int32_t *ids, int64_t M, int topk, double *y64,
                       double *bound)
{
    if (qt < 0 || qt >= T_COUNT || K % QK[qt] != 0) return -1;
    int64_t nb = K / QK[qt];
    int64_t rowbytes = nb * QB[qt];
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t t = 0; t < M; t++) {
        for (int j = 0; j < topk; j++) {
            int32_t e = ids[t * topk + j];
            double *w = (double *)malloc((size_t)K * sizeof(double));
            for (int64_t n = 0; n < N; n++) {
                int64_t o = (t * topk + j) * N + n;
                if (e < 0 || e >= E) {
                    if (y64) y64[o] = NAN;
                    if (bound) bound[o] = NAN;
                    continue;
                }
                orc_dequant_f64(qt, wq[e] + n * rowbytes, 1, K, w);
                double s = 0.0, a = 0.0;
                for (int64_t k = 0; k < K; k++) {
                    double pr = w[k] * x_at(x, xbf16, (x_per_slot ? t * topk + j : t) * K + k);
                    s += pr;
                    a += fabs(pr);
                }
                if (y64) y64[o] = s;
                if (bound) bound[o] = a;
            }
            free(w);
        }
    }
    return 0;
}

int orc_qmm_id(int qt, int xbf16, const uint8_t *const *wq, int64_t E, int64_t N, int64_t K, const void *x,
               const int32_t *ids, int64_t M, int topk, double *y64, double *bound)
{
    return qmm_id_rows(qt, xbf16, wq, E, N, K, x, 0, ids, M, topk, y64, bound);
}

/* The same with one activation row per (token, slot): x is M x topk x K. */
int orc_qmm_id_slots(int qt, int xbf16, const uint8_t *const *wq, int64_t E, int64_t N, int64_t K,
                     const void *x, const int32_t *ids, int64_t M, int topk, double *y64, double *bound)
{
    return qmm_id_rows(qt, xbf16, wq, E, N, K, x, 1, ids, M, topk, y64, bound);
}
