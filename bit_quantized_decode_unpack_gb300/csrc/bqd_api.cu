// Host side of the C ABI: argument validation and dispatch by format and M
// (the routing rules of "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析",
// §二 and §三: route by bit width and by the number of activation rows).
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "bqd_internal.cuh"

namespace bqd {

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

// Process-wide options (bqd_set_option).  The environment supplies their
// first values -- BQD_FORCE_KERNEL=generic|mma|tma|qmm, BQD_T5_STAGES=1|2,
// BQD_DEBUG_PLAN -- read once, on first use; afterwards only
// bqd_set_option changes them, so no call pays for reading the environment.
namespace {
struct Options {
    std::atomic<int> kernel{BQD_KERNEL_AUTO};
    std::atomic<int> t5_stages{0};
    std::atomic<int> debug_plan{0};
    std::atomic<int64_t> wait_ns{kDefaultWaitNs};
    Options()
    {
        if (const char *v = getenv("BQD_FORCE_KERNEL")) {
            if (strcmp(v, "generic") == 0) kernel = BQD_KERNEL_GENERIC;
            else if (strcmp(v, "mma") == 0) kernel = BQD_KERNEL_MMA;
            else if (strcmp(v, "tma") == 0) kernel = BQD_KERNEL_TMA;
            else if (strcmp(v, "qmm") == 0) kernel = BQD_KERNEL_QMM;
        }
        if (const char *v = getenv("BQD_T5_STAGES")) {
            const int n = atoi(v);
            t5_stages = (n == 1 || n == 2) ? n : 0;
        }
        debug_plan = getenv("BQD_DEBUG_PLAN") != nullptr;
    }
};
Options &options()
{
    static Options o;  // initialised once, thread-safely
    return o;
}
}  // namespace

int opt_kernel() { return options().kernel.load(std::memory_order_relaxed); }
int opt_t5_stages() { return options().t5_stages.load(std::memory_order_relaxed); }
bool opt_debug_plan() { return options().debug_plan.load(std::memory_order_relaxed) != 0; }
uint64_t opt_wait_ns() { return (uint64_t)options().wait_ns.load(std::memory_order_relaxed); }

}  // namespace bqd

using namespace bqd;

static bool valid_format(int f) { return f == BQD_FMT_AFFINE1 || f == BQD_FMT_AFFINE2 || f == BQD_FMT_T5; }
static bool valid_gs(int gs) { return gs == 64 || gs == 128; }
static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// N*K and M*K must stay far from int64 overflow; 2^50 elements is far beyond
// any device memory.
static bool sane(int64_t a, int64_t b) { return a >= 0 && b >= 0 && (a == 0 || b <= (int64_t(1) << 50) / a); }

extern "C" int bqd_abi_version(void) { return BQD_ABI_VERSION; }

extern "C" const char *bqd_status_string(int status)
{
    switch (status) {
    case BQD_OK: return "ok";
    case BQD_ERR_INVALID_ARG: return "invalid argument";
    case BQD_ERR_UNSUPPORTED: return "unsupported request";
    case BQD_ERR_ALIGNMENT: return "pointer alignment below the documented minimum";
    case BQD_ERR_BAD_T5_BYTE: return "invalid t5 byte (>= 243 or non-zero padding trit)";
    case BQD_ERR_NOT_TERNARY: return "2-bit code 3 where a ternary code was required";
    case BQD_ERR_CUDA: return "CUDA runtime or launch error";
    case BQD_ERR_TIMEOUT: return "bounded device-side wait expired";
    case BQD_ERR_ABI: return "ABI version mismatch";
    default: return "unknown status";
    }
}

extern "C" size_t bqd_packed_bytes(int format, int64_t N, int64_t K, int group_size)
{
    if (!valid_format(format) || !valid_gs(group_size) || !sane(N, K) || K % group_size != 0)
        return 0;
    return (size_t)(N * row_bytes_of(format, K, group_size));
}

static int qmv_common(const void *x, const void *w, const void *scales, const void *biases,
                      float ratio, int64_t M, int64_t N, int64_t K, int format, int gs,
                      void *out, bqd_stream_t stream)
{
    if (!valid_format(format) || !valid_gs(gs)) return BQD_ERR_INVALID_ARG;
    if (!sane(M, K) || !sane(N, K) || !sane(M, N) || K % gs != 0) return BQD_ERR_INVALID_ARG;
    if (!(ratio == ratio) || ratio > 3.0e38f || ratio < -3.0e38f) return BQD_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BQD_OK;
    if (!out) return BQD_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return BQD_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return cuda_status(cudaMemsetAsync(out, 0, (size_t)(M * N) * sizeof(__half), s));
    if (!x || !w || !scales) return BQD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(scales, 2) || (biases && !aligned(biases, 2)))
        return BQD_ERR_ALIGNMENT;

    QmvArgs a;
    a.x = static_cast<const __half *>(x);
    a.w = static_cast<const uint8_t *>(w);
    a.scales = static_cast<const __half *>(scales);
    a.biases = static_cast<const __half *>(biases);
    a.ratio = ratio;
    a.M = M; a.N = N; a.K = K; a.G = K / gs;
    a.fmt = format; a.gs = gs;
    a.row_bytes = row_bytes_of(format, K, gs);
    a.out = static_cast<__half *>(out);

    const int force = opt_kernel();
    if (force != 1) {
        // prefill: fused unpack + tcgen05 matrix product.  Below these sizes the
        // decode kernels (all passes of their x rows in one launch) are faster
        // (measured on a 27B-class layer): the product's 128-row tiles need a
        // wide N (gate/up: 136 tiles; down: 40) to fill the GPU at small M.
        // t5 (8 rows per decode pass): wide layers from M = 17 (gate gs128:
        // 36.3 us against 29.0 for two passes at M = 9..16; three passes
        // cost more), the long-K down projection from M = 25 (24 rows: 66.5
        // against 63.1; 32 rows: 66.6 against 85.3), narrower layers from
        // M = 33 (5120 x 5120 at 32 rows: 37.4 against 30.8)
        const bool wide = N >= 8192;
        const bool prefill = format == BQD_FMT_T5 ? (wide ? M > 16 : (K >= 8192 ? M > 24 : M > 32))
                                                  : (wide ? M > (format == BQD_FMT_AFFINE2 ? 16 : 32) : M > 64);
        if ((prefill && force != 3) || force == 4) {
            int st = launch_qmm(a, s);
            if (st != BQD_ERR_UNSUPPORTED || force == 2 || force == 4) return st;
        }
        if (force != 2) {
            // TMA-ring kernels (1/2-bit: K a multiple of 256; t5: of 1024;
            // aligned rows and bases)
            int st = format == BQD_FMT_T5 ? launch_qmv_t5r(a, s) : launch_qmv_tma(a, s);
            if (st != BQD_ERR_UNSUPPORTED || force == 3) return st;
        }
        int st = format == BQD_FMT_T5 ? launch_qmv_t5(a, s) : launch_qmv_mma(a, s);
        if (st != BQD_ERR_UNSUPPORTED || force == 2) return st;
    }
    return launch_qmv_generic(a, s);
}

static float default_ratio(int format)
{
    return format == BQD_FMT_AFFINE1 ? 0.5f : (format == BQD_FMT_AFFINE2 ? 1.5f : 1.0f);
}

extern "C" int bqd_qmv(const void *x, const void *w_packed, const void *scales, const void *biases,
                       int64_t M, int64_t N, int64_t K, int format, int group_size, void *out,
                       bqd_stream_t stream)
{
    return qmv_common(x, w_packed, scales, biases, default_ratio(format), M, N, K, format,
                      group_size, out, stream);
}

extern "C" int bqd_qmv_sym(const void *x, const void *w_packed, const void *scales, float ratio,
                           int64_t M, int64_t N, int64_t K, int format, int group_size, void *out,
                           bqd_stream_t stream)
{
    return qmv_common(x, w_packed, scales, nullptr, ratio, M, N, K, format, group_size, out, stream);
}

extern "C" int bqd_spec_decode_verify(const void *logits, int dtype, const int32_t *draft, int64_t B, int64_t D,
                                      int64_t V, int32_t *accepted, int32_t *next_token, int32_t *argmax_out,
                                      bqd_stream_t stream)
{
    if (dtype != BQD_DTYPE_F16 && dtype != BQD_DTYPE_F32) return BQD_ERR_INVALID_ARG;
    if (B < 0 || B > ((int64_t)1 << 26) || D < 0 || D > 4095 || V < 1 || V > ((int64_t)1 << 31) - 1024)
        return BQD_ERR_INVALID_ARG;
    if (B == 0) return BQD_OK;
    if (!logits || !accepted || !next_token || (D > 0 && !draft)) return BQD_ERR_INVALID_ARG;
    if (!aligned(logits, dtype == BQD_DTYPE_F16 ? 2 : 4) || !aligned(accepted, 4) || !aligned(next_token, 4) ||
        (draft && !aligned(draft, 4)) || (argmax_out && !aligned(argmax_out, 4)))
        return BQD_ERR_ALIGNMENT;
    return launch_spec_decode_verify(logits, dtype, draft, B, D, V, accepted, next_token, argmax_out,
                                     reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int bqd_pack(const uint8_t *codes, int64_t N, int64_t K, int format, int group_size,
                        void *w_packed, bqd_stream_t stream)
{
    if (!valid_format(format) || !valid_gs(group_size) || !sane(N, K) || K % group_size != 0)
        return BQD_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return BQD_OK;
    if (!codes || !w_packed) return BQD_ERR_INVALID_ARG;
    if (format != BQD_FMT_T5 && !aligned(w_packed, 4)) return BQD_ERR_ALIGNMENT;
    return launch_pack(codes, N, K, format, group_size, static_cast<uint8_t *>(w_packed),
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int bqd_unpack(const void *w_packed, int64_t N, int64_t K, int format, int group_size,
                          uint8_t *codes, bqd_stream_t stream)
{
    if (!valid_format(format) || !valid_gs(group_size) || !sane(N, K) || K % group_size != 0)
        return BQD_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return BQD_OK;
    if (!codes || !w_packed) return BQD_ERR_INVALID_ARG;
    if (format != BQD_FMT_T5 && !aligned(w_packed, 4)) return BQD_ERR_ALIGNMENT;
    return launch_unpack(static_cast<const uint8_t *>(w_packed), N, K, format, group_size, codes,
                         reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int bqd_repack_2bit_to_t5(const void *w2, int64_t N, int64_t K, int group_size,
                                     uint8_t *w_t5, int *d_status, bqd_stream_t stream)
{
    if (!valid_gs(group_size) || !sane(N, K) || K % group_size != 0) return BQD_ERR_INVALID_ARG;
    if (!d_status) return BQD_ERR_INVALID_ARG;
    if (!aligned(d_status, 4)) return BQD_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0 || K == 0) return cuda_status(cudaMemsetAsync(d_status, 0, sizeof(int), s));
    if (!w2 || !w_t5) return BQD_ERR_INVALID_ARG;
    if (!aligned(w2, 4)) return BQD_ERR_ALIGNMENT;
    return launch_repack_2bit_to_t5(static_cast<const uint8_t *>(w2), N, K, group_size, w_t5,
                                    d_status, s);
}

extern "C" int bqd_validate_t5(const uint8_t *w_t5, int64_t N, int64_t K, int group_size,
                               int *d_status, bqd_stream_t stream)
{
    if (!valid_gs(group_size) || !sane(N, K) || K % group_size != 0) return BQD_ERR_INVALID_ARG;
    if (!d_status) return BQD_ERR_INVALID_ARG;
    if (!aligned(d_status, 4)) return BQD_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0 || K == 0) return cuda_status(cudaMemsetAsync(d_status, 0, sizeof(int), s));
    if (!w_t5) return BQD_ERR_INVALID_ARG;
    return launch_validate_t5(w_t5, N, K, group_size, d_status, s);
}

extern "C" int bqd_detect_sym(const void *scales, const void *biases, int64_t N, int64_t G,
                              float ratio, int *d_mismatches, bqd_stream_t stream)
{
    if (!sane(N, G) || !d_mismatches) return BQD_ERR_INVALID_ARG;
    if (!(ratio == ratio) || ratio > 3.0e38f || ratio < -3.0e38f) return BQD_ERR_INVALID_ARG;
    if (!aligned(d_mismatches, 4)) return BQD_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0 || G == 0) return cuda_status(cudaMemsetAsync(d_mismatches, 0, sizeof(int), s));
    if (!scales || !biases) return BQD_ERR_INVALID_ARG;
    if (!aligned(scales, 2) || !aligned(biases, 2)) return BQD_ERR_ALIGNMENT;
    return launch_detect_sym(static_cast<const __half *>(scales), static_cast<const __half *>(biases),
                             N * G, ratio, d_mismatches, s);
}

extern "C" int bqd_device_status(bqd_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return BQD_ERR_CUDA;
    unsigned int n1 = 0, n2 = 0, n3 = 0, n4 = 0, n5 = 0;
    int st = take_qmv_mma_timeouts(&n1);
    if (st != BQD_OK) return st;
    st = take_qmv_t5_timeouts(&n2);
    if (st != BQD_OK) return st;
    st = take_qmm_timeouts(&n3);
    if (st != BQD_OK) return st;
    st = take_qmv_tma_timeouts(&n4);
    if (st != BQD_OK) return st;
    st = take_qmv_t5r_timeouts(&n5);
    if (st != BQD_OK) return st;
    return (n1 || n2 || n3 || n4 || n5) ? BQD_ERR_TIMEOUT : BQD_OK;
}

extern "C" int bqd_set_option(int option, int64_t value)
{
    Options &o = options();
    switch (option) {
    case BQD_OPT_KERNEL:
        if (value < BQD_KERNEL_AUTO || value > BQD_KERNEL_QMM) return BQD_ERR_INVALID_ARG;
        o.kernel = (int)value;
        return BQD_OK;
    case BQD_OPT_T5_STAGES:
        if (value < 0 || value > 2) return BQD_ERR_INVALID_ARG;
        o.t5_stages = (int)value;
        return BQD_OK;
    case BQD_OPT_DEBUG_PLAN:
        o.debug_plan = value != 0;
        return BQD_OK;
    case BQD_OPT_WAIT_LIMIT_NS:
        if (value < 0) return BQD_ERR_INVALID_ARG;
        o.wait_ns = value == 0 ? kDefaultWaitNs : value;
        return BQD_OK;
    default:
        return BQD_ERR_INVALID_ARG;
    }
}

extern "C" int64_t bqd_get_option(int option)
{
    switch (option) {
    case BQD_OPT_KERNEL: return opt_kernel();
    case BQD_OPT_T5_STAGES: return opt_t5_stages();
    case BQD_OPT_DEBUG_PLAN: return opt_debug_plan() ? 1 : 0;
    case BQD_OPT_WAIT_LIMIT_NS: return (int64_t)opt_wait_ns();
    default: return -1;
    }
}
