// Internal declarations shared by the libbqd translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bqd.h"

namespace bqd {

// One QMV request after host validation.  Pointers are device pointers.
struct QmvArgs {
    const __half *x;       // [M, K]
    const uint8_t *w;      // packed, row pitch = row_bytes
    const __half *scales;  // [N, G]
    const __half *biases;  // [N, G] or nullptr (sym)
    float ratio;           // sym ratio, used when biases == nullptr
    int64_t M, N, K, G, row_bytes;
    int fmt, gs;
    __half *out;           // [M, N]
};

inline int64_t t5_bytes_per_group(int gs) { return (gs + 4) / 5; }

inline int64_t row_bytes_of(int fmt, int64_t K, int gs)
{
    if (fmt == BQD_FMT_AFFINE1) return K / 8;
    if (fmt == BQD_FMT_AFFINE2) return K / 4;
    return (K / gs) * t5_bytes_per_group(gs);
}

// Kernel launchers (return a BQD_* status).
int launch_qmv_generic(const QmvArgs &a, cudaStream_t s);
// Tensor-core decode path; BQD_ERR_UNSUPPORTED when the request is outside
// its shape/alignment envelope (the caller then uses the generic kernel).
int launch_qmv_mma(const QmvArgs &a, cudaStream_t s);
// Tensor-core decode path for 1/2-bit codes fed by a TMA shared-memory ring
// (K a multiple of 256, K/gs a multiple of 8, 16-byte aligned rows and
// bases); same contract.
int launch_qmv_tma(const QmvArgs &a, cudaStream_t s);
// Tensor-core decode path for t5 weights fed by a TMA shared-memory ring (K a
// multiple of 1024, K/gs a multiple of 8, 16-byte aligned bases); same contract.
int launch_qmv_t5r(const QmvArgs &a, cudaStream_t s);
// Tensor-core decode path for t5 weights (K a multiple of 1024); same contract.
int launch_qmv_t5(const QmvArgs &a, cudaStream_t s);
// Prefill matrix product on tcgen05 tensor cores (for prefill-sized M), every
// format (16-byte aligned weight base; t5 rows a multiple of 16 bytes).
int launch_qmm(const QmvArgs &a, cudaStream_t s);

// Speculative-decoding verification (validated arguments, B >= 1).
int launch_spec_decode_verify(const void *logits, int dtype, const int32_t *draft, int64_t B, int64_t D, int64_t V,
                              int32_t *accepted, int32_t *next_token, int32_t *argmax_out, cudaStream_t s);

int launch_pack(const uint8_t *codes, int64_t N, int64_t K, int fmt, int gs,
                uint8_t *w, cudaStream_t s);
int launch_unpack(const uint8_t *w, int64_t N, int64_t K, int fmt, int gs,
                  uint8_t *codes, cudaStream_t s);
int launch_repack_2bit_to_t5(const uint8_t *w2, int64_t N, int64_t K, int gs,
                             uint8_t *w5, int *d_status, cudaStream_t s);
int launch_validate_t5(const uint8_t *w5, int64_t N, int64_t K, int gs,
                       int *d_status, cudaStream_t s);
int launch_detect_sym(const __half *scales, const __half *biases, int64_t count,
                      float ratio, int *d_mismatches, cudaStream_t s);

// Sym bias rebuilt from a scale: fp16_rne(float(-ratio) * float(scale)).
__device__ __forceinline__ __half sym_bias(__half s, float ratio)
{
    return __float2half_rn(__fmul_rn(-ratio, __half2float(s)));
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? BQD_OK : BQD_ERR_CUDA; }

// Reads and clears the counter of expired bounded waits of the tensor-core
// decode kernel; BQD_OK / BQD_ERR_CUDA.
int take_qmv_mma_timeouts(unsigned int *count);
int take_qmv_t5_timeouts(unsigned int *count);
int take_qmm_timeouts(unsigned int *count);
int take_qmv_tma_timeouts(unsigned int *count);
int take_qmv_t5r_timeouts(unsigned int *count);

// Number of SMs of the current device (cached per device).
int sm_count();

// Process-wide options (bqd_set_option; first values from the environment,
// read once).
constexpr int64_t kDefaultWaitNs = 1000000000;  // a bounded wait gives up after 1 s
int opt_kernel();         // BQD_KERNEL_*
int opt_t5_stages();      // 0 = planner's choice, else 1 or 2 (register-streaming t5 kernel)
bool opt_debug_plan();    // print each launch plan to stderr
uint64_t opt_wait_ns();   // limit of the ring kernels' pipeline waits, ns

}  // namespace bqd
