// Layout kernels: pack / unpack, 2-bit -> t5 repack, t5 validation and the
// load-time sym (identity I-B) check.  Page: "oMLX Bonsai 自定义内核:Qwen 系列
// 快速 QMV 路径完整解析" -- §二.1 (1-bit codes, 32 per uint32), §二.2 (I-B:
// bias = -scale*ratio), §二.3 (t5: trits {0,1,2}, 13/26 bytes per group; the
// repack_ternary_t5 tool; loading uint8 t5 weights).
#include "bqd_internal.cuh"

namespace bqd {
namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t work)
{
    int64_t blocks = (work + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)sm_count() * 16;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

__device__ __forceinline__ int t5_bytes(int gs) { return (gs + 4) / 5; }

// One thread per output uint32: BITS-bit codes, LSB first.
template <int BITS>
__global__ void pack_words_kernel(const uint8_t *__restrict__ codes, int64_t total_words,
                                  uint32_t *__restrict__ w)
{
    constexpr int per_word = 32 / BITS;
    constexpr uint32_t mask = (1u << BITS) - 1u;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total_words;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t *c = codes + i * per_word;  // rows are contiguous: K % per_word == 0
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < per_word; ++j) v |= (uint32_t(c[j]) & mask) << (BITS * j);
        w[i] = v;
    }
}

// One thread per output t5 byte.
__global__ void pack_t5_kernel(const uint8_t *__restrict__ codes, int64_t N, int64_t K, int gs,
                               uint8_t *__restrict__ w)
{
    const int B = t5_bytes(gs);
    const int64_t rb = (K / gs) * B;
    const int64_t total = N * rb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / rb, p = i % rb;
        const int64_t g = p / B;
        const int pin = (int)(p % B);
        const uint8_t *c = codes + n * K + g * gs;
        int v = 0, pw = 1;
        for (int d = 0; d < 5; ++d) {
            const int within = 5 * pin + d;
            if (within < gs) {
                int t = c[within];
                v += (t > 2 ? 0 : t) * pw;
            }
            pw *= 3;
        }
        w[i] = (uint8_t)v;
    }
}

// One thread per code.
__global__ void unpack_kernel(const uint8_t *__restrict__ w, int64_t N, int64_t K, int fmt, int gs,
                              uint8_t *__restrict__ codes)
{
    const int64_t total = N * K;
    const int B = t5_bytes(gs);
    const int64_t rb = fmt == BQD_FMT_AFFINE1 ? K / 8 : (fmt == BQD_FMT_AFFINE2 ? K / 4 : (K / gs) * B);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / K, k = i % K;
        const uint8_t *row = w + n * rb;
        int code;
        if (fmt == BQD_FMT_AFFINE1) {
            uint32_t word = reinterpret_cast<const uint32_t *>(row)[k >> 5];
            code = (word >> (k & 31)) & 1u;
        } else if (fmt == BQD_FMT_AFFINE2) {
            uint32_t word = reinterpret_cast<const uint32_t *>(row)[k >> 4];
            code = (word >> (2 * (k & 15))) & 3u;
        } else {
            const int64_t g = k / gs;
            const int within = (int)(k % gs);
            int v = row[g * B + within / 5];
            for (int d = within % 5; d > 0; --d) v /= 3;
            code = v % 3;
        }
        codes[i] = (uint8_t)code;
    }
}

// One thread per t5 byte, reading its (up to) five 2-bit codes.
__global__ void repack_kernel(const uint32_t *__restrict__ w2, int64_t N, int64_t K, int gs,
                              uint8_t *__restrict__ w5, int *__restrict__ status)
{
    const int B = t5_bytes(gs);
    const int64_t rb = (K / gs) * B;
    const int64_t total = N * rb;
    const int64_t words_per_row = K / 16;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / rb, p = i % rb;
        const int64_t g = p / B;
        const int pin = (int)(p % B);
        int v = 0, pw = 1, bad = 0;
        for (int d = 0; d < 5; ++d) {
            const int within = 5 * pin + d;
            if (within < gs) {
                const int64_t k = g * gs + within;
                int q = (w2[n * words_per_row + (k >> 4)] >> (2 * (k & 15))) & 3u;
                if (q == 3) {
                    ++bad;
                    q = 0;
                }
                v += q * pw;
            }
            pw *= 3;
        }
        w5[i] = (uint8_t)v;
        if (bad) atomicAdd(status, bad);
    }
}

// One thread per t5 byte.
__global__ void validate_t5_kernel(const uint8_t *__restrict__ w5, int64_t total, int gs,
                                   int *__restrict__ status)
{
    const int B = t5_bytes(gs);
    const int live = gs - 5 * (B - 1);  // trits used by a group's last byte
    int limit = 1;
    for (int d = 0; d < live; ++d) limit *= 3;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int v = w5[i];
        // rows hold whole groups, so (i % B) locates the byte within its group
        const bool last = (i % B) == B - 1;
        if (v >= 243 || (last && v >= limit)) atomicAdd(status, 1);
    }
}

__global__ void detect_sym_kernel(const __half *__restrict__ s, const __half *__restrict__ b,
                                  int64_t total, float ratio, int *__restrict__ mismatches)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const __half r = sym_bias(s[i], ratio);
        if (__half_as_ushort(r) != __half_as_ushort(b[i])) atomicAdd(mismatches, 1);
    }
}

}  // namespace

int launch_pack(const uint8_t *codes, int64_t N, int64_t K, int fmt, int gs, uint8_t *w,
                cudaStream_t s)
{
    if (fmt == BQD_FMT_AFFINE1) {
        const int64_t words = N * K / 32;
        pack_words_kernel<1><<<grid_for(words), kThreads, 0, s>>>(codes, words, reinterpret_cast<uint32_t *>(w));
    } else if (fmt == BQD_FMT_AFFINE2) {
        const int64_t words = N * K / 16;
        pack_words_kernel<2><<<grid_for(words), kThreads, 0, s>>>(codes, words, reinterpret_cast<uint32_t *>(w));
    } else {
        pack_t5_kernel<<<grid_for(N * (K / gs) * t5_bytes_per_group(gs)), kThreads, 0, s>>>(codes, N, K, gs, w);
    }
    return cuda_status(cudaGetLastError());
}

int launch_unpack(const uint8_t *w, int64_t N, int64_t K, int fmt, int gs, uint8_t *codes,
                  cudaStream_t s)
{
    unpack_kernel<<<grid_for(N * K), kThreads, 0, s>>>(w, N, K, fmt, gs, codes);
    return cuda_status(cudaGetLastError());
}

int launch_repack_2bit_to_t5(const uint8_t *w2, int64_t N, int64_t K, int gs, uint8_t *w5,
                             int *d_status, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(int), s);
    if (e != cudaSuccess) return BQD_ERR_CUDA;
    repack_kernel<<<grid_for(N * (K / gs) * t5_bytes_per_group(gs)), kThreads, 0, s>>>(
        reinterpret_cast<const uint32_t *>(w2), N, K, gs, w5, d_status);
    return cuda_status(cudaGetLastError());
}

int launch_validate_t5(const uint8_t *w5, int64_t N, int64_t K, int gs, int *d_status,
                       cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(int), s);
    if (e != cudaSuccess) return BQD_ERR_CUDA;
    const int64_t total = N * (K / gs) * t5_bytes_per_group(gs);
    validate_t5_kernel<<<grid_for(total), kThreads, 0, s>>>(w5, total, gs, d_status);
    return cuda_status(cudaGetLastError());
}

int launch_detect_sym(const __half *scales, const __half *biases, int64_t count, float ratio,
                      int *d_mismatches, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(d_mismatches, 0, sizeof(int), s);
    if (e != cudaSuccess) return BQD_ERR_CUDA;
    detect_sym_kernel<<<grid_for(count), kThreads, 0, s>>>(scales, biases, count, ratio, d_mismatches);
    return cuda_status(cudaGetLastError());
}

}  // namespace bqd
