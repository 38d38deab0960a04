/*
 * bqd.h -- C ABI of libbqd: the decode-time low-bit quantized matrix-vector
 * product (QMV), its prefill matrix product (QMM) and the speculative-decoding
 * verification kernel, on GB300 (sm_103a).
 *
 * Page defining the operations: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径
 * 完整解析" (oMLX Bonsai custom kernels: the fast QMV path for the Qwen
 * family), cnnetsun.cn/a/4328761.  Section numbers (§二.1 ...) are that page's.
 *
 * The product (§二.1, §二.2):
 *     y[m, n] = sum_k x[m, k] * (scale[n, k/gs] * q[n, k] + bias[n, k/gs])
 * for m < M activation rows, n < N weight rows (output features), k < K input
 * features, group size gs in {64, 128}, G = K / gs groups per row.
 *
 * Data layout (all tensors dense, row-major, no strides):
 *   x       fp16 [M, K]
 *   scales  fp16 [N, G]
 *   biases  fp16 [N, G], or NULL ("sym": bias = -ratio * scale, not read)
 *   out     fp16 [M, N]   (fp32 accumulation, rounded to nearest even)
 *   w_packed, row n at byte offset n * bqd_packed_bytes(format, 1, K, gs):
 *     BQD_FMT_AFFINE1: uint32 [N, K/32]; code k = 32j+i is bit i of word j
 *     BQD_FMT_AFFINE2: uint32 [N, K/16]; code k = 16j+i is bits 2i..2i+1
 *     BQD_FMT_T5     : uint8  [N, G*ceil(gs/5)]; trits {0,1,2}; byte p of a
 *                      group holds weights 5p..5p+4 of it as sum_i t_i 3^i
 *                      (first weight least significant); 13 bytes per
 *                      64-group, 26 per 128-group (§二.3); the unused high
 *                      trits of a group's last byte are 0
 *   Words are little-endian.
 *
 * Conventions for every entry point:
 *  - Pointers named d_* or documented as device pointers are device memory of
 *    the current CUDA device; the caller allocates, owns and frees them.  The
 *    library allocates no device memory per call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and return the status of argument validation plus kernel
 *    launch.  Errors found in the DATA (a bad t5 byte, a 2-bit code 3 where a
 *    ternary code is needed) are written to a caller-provided device counter,
 *    which the caller reads back after synchronising.  Kernels never trap.
 *  - Validation happens on the host before anything is enqueued: on an error
 *    nothing is launched and no output is touched.
 *  - Thread-safe and reentrant; calls on one stream run in order.
 */
#ifndef BQD_H
#define BQD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BQD_ABI_VERSION 1

/* status codes */
enum {
    BQD_OK = 0,
    BQD_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad format/group size */
    BQD_ERR_UNSUPPORTED = 2, /* valid request this build does not serve      */
    BQD_ERR_ALIGNMENT = 3,   /* pointer alignment below what is documented   */
    BQD_ERR_BAD_T5_BYTE = 4, /* (for callers mapping a validate count)       */
    BQD_ERR_NOT_TERNARY = 5, /* (for callers mapping a repack count)         */
    BQD_ERR_CUDA = 6,        /* a CUDA runtime call or a launch failed       */
    BQD_ERR_TIMEOUT = 7,     /* a bounded device-side wait ran out           */
    BQD_ERR_ABI = 8          /* header / library ABI mismatch                */
};

/* weight formats */
enum { BQD_FMT_AFFINE1 = 1, BQD_FMT_AFFINE2 = 2, BQD_FMT_T5 = 3 };

/* element types of bqd_spec_decode_verify's logits */
enum { BQD_DTYPE_F16 = 1, BQD_DTYPE_F32 = 2 };

/* opaque CUDA stream (binary-compatible with cudaStream_t / CUstream) */
typedef struct CUstream_st *bqd_stream_t;

/*
 * ABI probe (§三: the extension is probed before use).  Returns
 * BQD_ABI_VERSION of the built library; a caller compiled against another
 * header version must not call the rest.  Host-only, never fails.
 */
int bqd_abi_version(void);

/* Static, human-readable text for a status code.  Host-only. */
const char *bqd_status_string(int status);

/*
 * Bytes of the packed weight matrix for (format, N, K, group_size): N*K/8 for
 * 1-bit, N*K/4 for 2-bit, N*(K/gs)*ceil(gs/5) for t5 (13 or 26 bytes per
 * group, §二.3).  Returns 0 for an invalid request (K not a multiple of gs,
 * gs not 64/128, unknown format, negative sizes).  Host-only.
 */
size_t bqd_packed_bytes(int format, int64_t N, int64_t K, int group_size);

/*
 * Quantized matrix-vector / matrix product, §二.1 (M = 1, qmv_fast),
 * §二.2 (M = 2..5, qmv_wide: each packed weight byte is read once for all M
 * rows; sym variant with biases == NULL reads no bias tensor), §二.3 (t5
 * decode, and the fused unpack + tensor-core matrix product for prefill).
 * Any M >= 0 is accepted; the library picks the kernel (decode kernels for
 * small M, the fused product once M is large enough for it on the layer's
 * shape -- beyond 10 to 64 rows depending on format and N).
 *   x        device fp16 [M, K], 16-byte aligned
 *   w_packed device, layout above, 16-byte aligned
 *   scales   device fp16 [N, G], 2-byte aligned
 *   biases   device fp16 [N, G] or NULL.  NULL means the sym identity I-B of
 *            §二.2 with the format's default ratio: 0.5 (1-bit), 1.5 (2-bit),
 *            1.0 (t5: w = scale*t - scale); bias = fp16(-ratio * scale)
 *   out      device fp16 [M, N], 16-byte aligned; fully overwritten
 * M >= 0, N >= 0, K >= 0 with K % group_size == 0.  M == 0 or N == 0 is a
 * no-op; K == 0 writes zeros.  Returns BQD_OK, BQD_ERR_INVALID_ARG,
 * BQD_ERR_ALIGNMENT or BQD_ERR_CUDA.
 */
int bqd_qmv(const void *x, const void *w_packed, const void *scales,
            const void *biases, int64_t M, int64_t N, int64_t K, int format,
            int group_size, void *out, bqd_stream_t stream);

/*
 * Sym variant with an explicit ratio (§二.2 identity I-B: bias =
 * -scale * ratio; the bias tensor does not exist and is not read).  The bias
 * is rebuilt as fp16_rne(float(-ratio) * float(scale)).  Arguments and errors
 * as bqd_qmv; ratio must be finite.
 */
int bqd_qmv_sym(const void *x, const void *w_packed, const void *scales,
                float ratio, int64_t M, int64_t N, int64_t K, int format,
                int group_size, void *out, bqd_stream_t stream);

/*
 * Pack codes into the format's layout (the layout above; §二.1, §二.3).
 *   codes    device uint8 [N, K]; values must be < 2 (1-bit), < 4 (2-bit),
 *            < 3 (t5); larger values are masked (1/2-bit) or taken as 0 (t5)
 *   w_packed device output, bqd_packed_bytes(format, N, K, gs) bytes
 * Returns BQD_OK, BQD_ERR_INVALID_ARG or BQD_ERR_CUDA.
 */
int bqd_pack(const uint8_t *codes, int64_t N, int64_t K, int format,
             int group_size, void *w_packed, bqd_stream_t stream);

/* Inverse of bqd_pack: w_packed (device) -> codes uint8 [N, K] (device). */
int bqd_unpack(const void *w_packed, int64_t N, int64_t K, int format,
               int group_size, uint8_t *codes, bqd_stream_t stream);

/*
 * Repack a 2-bit matrix whose codes are ternary {0,1,2} into t5 (§二.3: the
 * repack_ternary_t5 tool).  The scales are unchanged; the caller's 2-bit
 * biases must equal -scale (t5 has no bias tensor) for the product to be
 * unchanged.
 *   w2       device, 2-bit layout [N, K/16] uint32
 *   w_t5     device output, bqd_packed_bytes(BQD_FMT_T5, N, K, gs) bytes
 *   d_status device int32: receives the number of 2-bit codes equal to 3
 *            (0 = success; otherwise the affected t5 bytes are unspecified).
 *            Reset to 0 by this call before counting.
 */
int bqd_repack_2bit_to_t5(const void *w2, int64_t N, int64_t K, int group_size,
                          uint8_t *w_t5, int *d_status, bqd_stream_t stream);

/*
 * Validate a t5 matrix (§二.3 load path accepting uint8 t5 weights).
 *   d_status device int32: receives the number of invalid bytes (>= 243, or a
 *            group's last byte with non-zero padding trits); reset to 0 by
 *            this call before counting.  The QMV/QMM kernels do not check
 *            bytes; their output for an invalid byte is unspecified.
 */
int bqd_validate_t5(const uint8_t *w_t5, int64_t N, int64_t K, int group_size,
                    int *d_status, bqd_stream_t stream);

/*
 * Load-time detection of identity I-B (§二.2): counts the (n, g) for which
 * biases[n,g] != fp16_rne(float(-ratio) * float(scales[n,g])), comparing
 * bit patterns.  A count of 0 means the bias tensor can be dropped and the
 * sym path used.
 *   scales, biases device fp16 [N, G];  d_mismatches device int32 (reset to 0
 *   by this call before counting).
 */
int bqd_detect_sym(const void *scales, const void *biases, int64_t N, int64_t G,
                   float ratio, int *d_mismatches, bqd_stream_t stream);

/*
 * Speculative-decoding verification in one kernel (§三: spec_decode_verify
 * fuses "compare the draft tokens -> count the accepted length -> produce the
 * correction token").  The page gives no formula; greedy reading:
 *   t[b, i]       = argmax over v of logits[b, i, v], i = 0 .. D (ties: the
 *                   smallest v; NaN entries are never chosen; a row of NaNs
 *                   gives -1)
 *   accepted[b]   = the largest a in [0, D] with draft[b, i] == t[b, i] for
 *                   every i < a (a -1 from a row of NaNs matches nothing)
 *   next_token[b] = t[b, accepted[b]]: the target's token where the draft was
 *                   first rejected, or the bonus token after D accepted drafts
 * Arguments (device pointers):
 *   logits      [B, D+1, V] of `dtype` (BQD_DTYPE_F16 or BQD_DTYPE_F32),
 *               aligned to its element size; row (b, i) scores the token
 *               that follows the prefix and draft[b, 0 .. i-1]
 *   draft       int32 [B, D] (may be NULL when D == 0); ids outside [0, V)
 *               never match
 *   accepted, next_token  int32 [B]
 *   argmax_out  int32 [B, D+1], or NULL: t[b, i] of every row
 * Sizes: 0 <= B <= 2^26, 0 <= D <= 4095, 1 <= V <= 2^31 - 1024.  B == 0
 * launches nothing.  Every logit is read once (the call is bound by HBM
 * bandwidth); one thread-block cluster of min(D+1, 16) CTAs per sequence.
 */
int bqd_spec_decode_verify(const void *logits, int dtype, const int32_t *draft, int64_t B, int64_t D,
                           int64_t V, int32_t *accepted, int32_t *next_token, int32_t *argmax_out,
                           bqd_stream_t stream);

/*
 * Device-side failure report.  Kernels that wait on asynchronous copies
 * (mbarrier waits) bound every wait; a wait that runs out makes that CTA skip
 * its work and bumps a library-owned device counter instead of hanging.  This
 * call synchronises `stream`, reads and clears that counter, and returns
 * BQD_ERR_TIMEOUT if any wait expired since the previous call (the outputs of
 * the affected calls are then unspecified), BQD_ERR_CUDA if the
 * synchronisation failed, else BQD_OK.  Host + device, blocking.
 */
int bqd_device_status(bqd_stream_t stream);

/*
 * Process-wide options: a control for tests and measurements, with no
 * counterpart on the page.  Host-only; a change applies to calls made after
 * it (calls already enqueued keep what they were launched with).
 *   BQD_OPT_KERNEL         BQD_KERNEL_AUTO (the dispatcher picks) or one
 *                          kernel family forced for every QMV call; a forced
 *                          family that cannot serve a request makes that call
 *                          return BQD_ERR_UNSUPPORTED instead of falling back
 *   BQD_OPT_T5_STAGES      0, or 1 / 2: the ring depth of the register-
 *                          streaming t5 kernel (0 = the planner's choice)
 *   BQD_OPT_WAIT_LIMIT_NS  time, in ns of %globaltimer, after which a pipeline
 *                          wait of the ring kernels gives up (see
 *                          bqd_device_status); 0 restores the default of 1 s.
 *                          The waits that let a CTA's own copies land before
 *                          it exits always keep the default limit
 *   BQD_OPT_DEBUG_PLAN     non-zero: print each launch plan to stderr
 * The environment gives the first values, read once on first use:
 * BQD_FORCE_KERNEL=generic|mma|tma|qmm, BQD_T5_STAGES=1|2, BQD_DEBUG_PLAN.
 * bqd_set_option returns BQD_OK or BQD_ERR_INVALID_ARG (unknown option or
 * value out of range); bqd_get_option returns the value, or -1 for an
 * unknown option.
 */
enum { BQD_OPT_KERNEL = 1, BQD_OPT_T5_STAGES = 2, BQD_OPT_WAIT_LIMIT_NS = 3, BQD_OPT_DEBUG_PLAN = 4 };
enum {
    BQD_KERNEL_AUTO = 0,    /* the dispatcher's choice                       */
    BQD_KERNEL_GENERIC = 1, /* CUDA-core kernel, any shape                   */
    BQD_KERNEL_MMA = 2,     /* register-streaming tensor-core decode kernels */
    BQD_KERNEL_TMA = 3,     /* TMA-ring decode kernels                       */
    BQD_KERNEL_QMM = 4      /* tcgen05 prefill product                       */
};
int bqd_set_option(int option, int64_t value);
int64_t bqd_get_option(int option);

#ifdef __cplusplus
}
#endif
#endif /* BQD_H */
