/*
 * bqd_oracle.c -- plain, slow, float64 CPU oracle.  TEST INFRASTRUCTURE ONLY
 * (tests, smoke check, benchmark CPU-baseline leg).  Written from the page
 * "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" (oMLX Bonsai custom
 * kernels: the fast QMV path for the Qwen family); see bqd_oracle.h for the
 * readings of the points that page leaves open.  No blocking, no fusion, no
 * reordering: every weight is decoded, dequantised and multiplied one by one.
 */
#include "bqd_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

/* ---- IEEE binary16, from the format's definition ------------------------ */

double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp_field = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (exp_field == 0) {
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-24 */
    } else if (exp_field == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), exp_field - 25); /* (1.m) * 2^(e-15) */
    }
    return sign ? -v : v;
}

uint16_t orc_float_to_half_rne(float f)
{
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0) /* at or above the midpoint 65504..65536: rounds to inf */
        return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: integer multiple of 2^-24, ties to even */
        double q = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q); /* q == 1024 encodes 2^-14 */
    }
    int e;
    frexp(a, &e);
    e -= 1; /* a = m * 2^e with m in [1, 2) */
    double q = rint(ldexp(a, 10 - e)); /* in [1024, 2048], ties to even */
    if (q >= 2048.0) {
        q = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31)
        return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* ---- packed layout ------------------------------------------------------ */

static int valid_fmt_gs(int fmt, int gs)
{
    if (gs != 64 && gs != 128)
        return 0;
    return fmt == ORC_FMT_AFFINE1 || fmt == ORC_FMT_AFFINE2 || fmt == ORC_FMT_T5;
}

static int64_t t5_bytes_per_group(int gs) { return (gs + 4) / 5; }

int64_t orc_row_bytes(int fmt, int64_t K, int gs)
{
    if (!valid_fmt_gs(fmt, gs) || K < 0 || K % gs != 0)
        return -1;
    if (fmt == ORC_FMT_AFFINE1)
        return (K / 32) * 4; /* one uint32 per 32 codes */
    if (fmt == ORC_FMT_AFFINE2)
        return (K / 16) * 4; /* one uint32 per 16 codes */
    return (K / gs) * t5_bytes_per_group(gs);
}

static uint32_t load_le32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

static void store_le32(uint8_t *p, uint32_t w)
{
    p[0] = (uint8_t)(w & 0xff);
    p[1] = (uint8_t)((w >> 8) & 0xff);
    p[2] = (uint8_t)((w >> 16) & 0xff);
    p[3] = (uint8_t)((w >> 24) & 0xff);
}

static int pow3(int i)
{
    int p = 1;
    while (i-- > 0)
        p *= 3;
    return p;
}

int orc_t5_encode(const uint8_t trits[5])
{
    int v = 0;
    for (int i = 0; i < 5; ++i)
        v += trits[i] * pow3(i);
    return v;
}

void orc_t5_decode(int byte_value, uint8_t trits[5])
{
    int v = byte_value;
    for (int i = 0; i < 5; ++i) {
        trits[i] = (uint8_t)(v % 3);
        v /= 3;
    }
}

int orc_code_at(const uint8_t *row, int fmt, int gs, int64_t k)
{
    if (fmt == ORC_FMT_AFFINE1) {
        uint32_t w = load_le32(row + 4 * (k / 32));
        return (int)((w >> (k % 32)) & 1u);
    }
    if (fmt == ORC_FMT_AFFINE2) {
        uint32_t w = load_le32(row + 4 * (k / 16));
        return (int)((w >> (2 * (k % 16))) & 3u);
    }
    /* t5 */
    int64_t g = k / gs, within = k % gs;
    int byte_value = row[g * t5_bytes_per_group(gs) + within / 5];
    return (byte_value / pow3((int)(within % 5))) % 3;
}

int64_t orc_pack(const uint8_t *codes, int64_t N, int64_t K, int fmt, int gs,
                 uint8_t *packed)
{
    int64_t rb = orc_row_bytes(fmt, K, gs);
    if (rb < 0 || N < 0)
        return -1;
    int max_code = fmt == ORC_FMT_AFFINE1 ? 1 : (fmt == ORC_FMT_AFFINE2 ? 3 : 2);
    int64_t bad = 0;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t *c = codes + n * K;
        uint8_t *row = packed + n * rb;
        memset(row, 0, (size_t)rb);
        for (int64_t k = 0; k < K; ++k)
            if (c[k] > max_code)
                ++bad;
        if (fmt == ORC_FMT_AFFINE1 || fmt == ORC_FMT_AFFINE2) {
            int bits = fmt == ORC_FMT_AFFINE1 ? 1 : 2;
            int per_word = 32 / bits;
            for (int64_t j = 0; j < K / per_word; ++j) {
                uint32_t w = 0;
                for (int i = 0; i < per_word; ++i) {
                    uint32_t code = c[j * per_word + i] & (uint32_t)max_code;
                    w |= code << (bits * i);
                }
                store_le32(row + 4 * j, w);
            }
        } else {
            int64_t B = t5_bytes_per_group(gs);
            for (int64_t g = 0; g < K / gs; ++g) {
                for (int64_t p = 0; p < B; ++p) {
                    uint8_t t[5] = {0, 0, 0, 0, 0};
                    for (int i = 0; i < 5; ++i) {
                        int64_t within = 5 * p + i;
                        if (within < gs) {
                            uint8_t code = c[g * gs + within];
                            t[i] = code > 2 ? 0 : code;
                        }
                    }
                    row[g * B + p] = (uint8_t)orc_t5_encode(t);
                }
            }
        }
    }
    return bad;
}

int64_t orc_unpack(const uint8_t *packed, int64_t N, int64_t K, int fmt, int gs,
                   uint8_t *codes)
{
    int64_t rb = orc_row_bytes(fmt, K, gs);
    if (rb < 0 || N < 0)
        return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)orc_code_at(packed + n * rb, fmt, gs, k);
    return 0;
}

int64_t orc_t5_invalid_bytes(const uint8_t *packed, int64_t N, int64_t K, int gs)
{
    int64_t rb = orc_row_bytes(ORC_FMT_T5, K, gs);
    if (rb < 0 || N < 0)
        return -1;
    int64_t B = t5_bytes_per_group(gs);
    int live_in_last = gs - 5 * (int)(B - 1); /* trits used by a group's last byte */
    int64_t bad = 0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < rb; ++i) {
            int v = packed[n * rb + i];
            if (v >= 243) {
                ++bad;
                continue;
            }
            if (i % B == B - 1) {
                uint8_t t[5];
                orc_t5_decode(v, t);
                for (int d = live_in_last; d < 5; ++d)
                    if (t[d] != 0) {
                        ++bad;
                        break;
                    }
            }
        }
    }
    return bad;
}

uint16_t orc_sym_bias(uint16_t scale_bits, double ratio)
{
    float s = (float)orc_half_to_double(scale_bits); /* exact */
    float prod = (float)(-ratio) * s;              /* rounded once, in float */
    return orc_float_to_half_rne(prod);
}

int64_t orc_sym_mismatches(const uint16_t *scales, const uint16_t *biases,
                           int64_t N, int64_t G, double ratio)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < N * G; ++i)
        if (orc_sym_bias(scales[i], ratio) != biases[i])
            ++bad;
    return bad;
}

int orc_qmv_rows(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                 const uint16_t *biases, double ratio, int64_t M, int64_t N,
                 int64_t K, int fmt, int gs, const int64_t *rows, int64_t nrows,
                 double *y, double *bound)
{
    int64_t rb = orc_row_bytes(fmt, K, gs);
    if (rb < 0 || M < 0 || N < 0 || nrows < 0)
        return -1;
    int64_t G = K / gs;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t n = rows[r];
        if (n < 0 || n >= N)
            return -1;
        const uint8_t *row = packed + n * rb;
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t g = k / gs;
                uint16_t sb = scales[n * G + g];
                double s = orc_half_to_double(sb);
                double b = biases ? orc_half_to_double(biases[n * G + g])
                                  : orc_half_to_double(orc_sym_bias(sb, ratio));
                double w = s * (double)orc_code_at(row, fmt, gs, k) + b;
                double p = orc_half_to_double(x[m * K + k]) * w;
                acc += p;
                mag += fabs(p);
            }
            y[m * nrows + r] = acc;
            bound[m * nrows + r] = mag;
        }
    }
    return 0;
}
