/*
 * bqd_oracle.h -- plain float64 CPU oracle for the low-bit quantized
 * matrix-vector product.  TEST INFRASTRUCTURE ONLY: only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Page followed: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析"
 * (oMLX Bonsai custom kernels: the fast QMV path for the Qwen family),
 * cnnetsun.cn/a/4328761.  Section numbers below (§二.1 ...) are that page's.
 *
 * Readings of points the page leaves open (each listed in the design notes):
 *  - Packing runs along K (the reduction axis), rows are contiguous
 *    (row-major [N, ...]), groups of `gs` consecutive k share one scale and
 *    one bias (§二.1 "affine" weights; group sizes 64/128 from §四).
 *  - 1-bit: 32 codes per uint32, LSB first: code k = 32j+i is bit i of word j
 *    (§二.1 "one uint32 holds 32 1-bit values ... unpacked by shifting").
 *  - 2-bit: 16 codes per uint32, LSB first: code k = 16j+i is bits 2i..2i+1.
 *  - Words are little-endian in memory.
 *  - t5: trits {0,1,2}, five per byte, byte = sum_i t_i * 3^i with the first
 *    weight least significant; each group starts on a fresh byte and takes
 *    ceil(gs/5) bytes (13 for gs=64, 26 for gs=128, §二.3); the unused high
 *    trits of a group's last byte are 0.  Bytes 243..255 are invalid.
 *  - Dequantised weight: w = scale*q + bias (affine).  When no bias tensor is
 *    given ("sym", §二.2 identity I-B: bias = -scale*ratio) the bias is
 *    rebuilt as fp16_rne(float(-ratio) * float(scale)).
 */
#ifndef BQD_ORACLE_H
#define BQD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_FMT_AFFINE1 = 1, ORC_FMT_AFFINE2 = 2, ORC_FMT_T5 = 3 };

/* IEEE binary16 bits -> exact double. */
double orc_half_to_double(uint16_t h);
/* float -> binary16 bits, round to nearest even (overflow -> inf). */
uint16_t orc_float_to_half_rne(float f);

/* Bytes of one packed row, or -1 for an invalid (fmt, K, gs). */
int64_t orc_row_bytes(int fmt, int64_t K, int gs);

/* Code of weight k in one packed row. */
int orc_code_at(const uint8_t *row, int fmt, int gs, int64_t k);

/* t5 byte <-> five trits (trit[0] least significant). */
int orc_t5_encode(const uint8_t trits[5]);
void orc_t5_decode(int byte_value, uint8_t trits[5]);

/* codes uint8 [N,K] <-> packed [N, row_bytes].  Return 0, or -1 on invalid
 * arguments, or the number of codes out of range for the format. */
int64_t orc_pack(const uint8_t *codes, int64_t N, int64_t K, int fmt, int gs,
                 uint8_t *packed);
int64_t orc_unpack(const uint8_t *packed, int64_t N, int64_t K, int fmt, int gs,
                   uint8_t *codes);

/* Number of invalid bytes in a t5 matrix: a byte >= 243, or a last byte of a
 * group whose padding trits are not 0.  -1 on invalid arguments. */
int64_t orc_t5_invalid_bytes(const uint8_t *packed, int64_t N, int64_t K, int gs);

/* Rebuilt sym bias for one scale (bits in, bits out). */
uint16_t orc_sym_bias(uint16_t scale_bits, double ratio);

/* Number of (n,g) whose stored bias differs from the rebuilt sym bias. */
int64_t orc_sym_mismatches(const uint16_t *scales, const uint16_t *biases,
                           int64_t N, int64_t G, double ratio);

/*
 * y[m, r] = sum_k x[m,k] * w[rows[r], k] in float64 for the listed rows,
 * with w = scale*q + bias.  bound[m, r] = sum_k |x[m,k] * w[rows[r], k]|.
 * x: fp16 bits [M, K]; scales/biases: fp16 bits [N, K/gs]; biases may be
 * NULL (sym, bias rebuilt from `ratio`).  y, bound: [M, nrows].
 * Returns 0, or -1 on invalid arguments.
 */
int orc_qmv_rows(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                 const uint16_t *biases, double ratio, int64_t M, int64_t N,
                 int64_t K, int fmt, int gs, const int64_t *rows, int64_t nrows,
                 double *y, double *bound);

#ifdef __cplusplus
}
#endif
#endif
