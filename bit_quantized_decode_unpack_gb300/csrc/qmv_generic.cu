// Generic QMV kernel: any format, any shape/alignment the ABI accepts.
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析", §二.1-§二.3.
// Computes y[m,n] = sum over the packed units u of row n of
//     s[n,g(u)] * sum_{k in u} q[n,k] x[m,k]  +  b[n,g(u)] * sum_{k in u} x[m,k]
// in fp32 on CUDA cores, where a unit is one uint32 word (1/2-bit; a word
// never straddles a group) or one t5 byte (five trits of one group).  One warp
// per weight row; consecutive lanes take consecutive units, so the activation
// loads of a warp are contiguous.  Codes are unpacked in registers (shifts
// for 1/2-bit, base-3 digits for t5); warp-shuffle reduction; fp16
// round-to-nearest-even store.  It serves the shapes the tensor-core decode
// kernel does not take and is the cross-check for that kernel.
#include "bqd_internal.cuh"

namespace bqd {
namespace {

constexpr int kWarps = 8;

template <int MT>
__device__ __forceinline__ void accumulate_unit(float (&acc)[MT], const float (&dot)[MT],
                                                const float (&sx)[MT], float s, float b)
{
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = fmaf(s, dot[m], fmaf(b, sx[m], acc[m]));
}

template <int FMT, int MT>
__global__ void __launch_bounds__(kWarps * 32)
qmv_generic_kernel(QmvArgs a, int64_t m0, int mrows)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int gs = a.gs;
    const int64_t K = a.K, G = a.G;
    const __half *xb = a.x + m0 * K;

    for (int64_t n = (int64_t)blockIdx.x * kWarps + warp; n < a.N; n += (int64_t)gridDim.x * kWarps) {
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        const uint8_t *row = a.w + n * a.row_bytes;
        const __half *srow = a.scales + n * G;
        const __half *brow = a.biases ? a.biases + n * G : nullptr;

        if (FMT == BQD_FMT_AFFINE1 || FMT == BQD_FMT_AFFINE2) {
            constexpr int bits = FMT == BQD_FMT_AFFINE1 ? 1 : 2;
            constexpr int per_word = 32 / bits;
            constexpr uint32_t mask = (1u << bits) - 1u;
            const int64_t words = K / per_word;
            const uint32_t *wp = reinterpret_cast<const uint32_t *>(row);
            for (int64_t j = lane; j < words; j += 32) {
                const uint32_t word = wp[j];
                const int64_t k0 = j * per_word;
                const int64_t g = k0 / gs;
                const __half sh = srow[g];
                const float s = __half2float(sh);
                const float b = __half2float(brow ? brow[g] : sym_bias(sh, a.ratio));
                float dot[MT], sx[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) dot[m] = sx[m] = 0.f;
#pragma unroll
                for (int v = 0; v < per_word / 8; ++v) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < mrows) {
                            const uint4 xv = *reinterpret_cast<const uint4 *>(xb + m * K + k0 + 8 * v);
                            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                __half2 x2;
                                *reinterpret_cast<uint32_t *>(&x2) = xw[h];
                                const float2 xf = __half22float2(x2);
                                const int i = 8 * v + 2 * h;
                                const float q0 = (float)((word >> (bits * i)) & mask);
                                const float q1 = (float)((word >> (bits * (i + 1))) & mask);
                                dot[m] = fmaf(q0, xf.x, fmaf(q1, xf.y, dot[m]));
                                sx[m] += xf.x + xf.y;
                            }
                        }
                    }
                }
                accumulate_unit<MT>(acc, dot, sx, s, b);
            }
        } else {
            const int B = (gs + 4) / 5;
            const int64_t nbytes = a.row_bytes;
            for (int64_t p = lane; p < nbytes; p += 32) {
                const int64_t g = p / B;
                const int pb = (int)(p % B);
                const __half sh = srow[g];
                const float s = __half2float(sh);
                const float b = __half2float(brow ? brow[g] : sym_bias(sh, a.ratio));
                int v = row[p];
                float dot[MT], sx[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) dot[m] = sx[m] = 0.f;
#pragma unroll
                for (int d = 0; d < 5; ++d) {
                    const int within = 5 * pb + d;
                    const float q = (float)(v % 3);
                    v /= 3;
                    if (within < gs) {
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (m < mrows) {
                                const float xv = __half2float(xb[m * K + g * gs + within]);
                                dot[m] = fmaf(q, xv, dot[m]);
                                sx[m] += xv;
                            }
                        }
                    }
                }
                accumulate_unit<MT>(acc, dot, sx, s, b);
            }
        }

#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < mrows) a.out[(m0 + m) * a.N + n] = __float2half_rn(acc[m]);
        }
    }
}

template <int FMT>
int launch_fmt(const QmvArgs &a, cudaStream_t s)
{
    const int64_t blocks_needed = (a.N + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)sm_count() * 8;
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    for (int64_t m0 = 0; m0 < a.M; m0 += 8) {
        const int mrows = (int)((a.M - m0) < 8 ? (a.M - m0) : 8);
        if (mrows == 1)
            qmv_generic_kernel<FMT, 1><<<grid, kWarps * 32, 0, s>>>(a, m0, mrows);
        else if (mrows == 2)
            qmv_generic_kernel<FMT, 2><<<grid, kWarps * 32, 0, s>>>(a, m0, mrows);
        else if (mrows <= 4)
            qmv_generic_kernel<FMT, 4><<<grid, kWarps * 32, 0, s>>>(a, m0, mrows);
        else
            qmv_generic_kernel<FMT, 8><<<grid, kWarps * 32, 0, s>>>(a, m0, mrows);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return BQD_ERR_CUDA;
    }
    return BQD_OK;
}

}  // namespace

int launch_qmv_generic(const QmvArgs &a, cudaStream_t s)
{
    switch (a.fmt) {
    case BQD_FMT_AFFINE1: return launch_fmt<BQD_FMT_AFFINE1>(a, s);
    case BQD_FMT_AFFINE2: return launch_fmt<BQD_FMT_AFFINE2>(a, s);
    case BQD_FMT_T5: return launch_fmt<BQD_FMT_T5>(a, s);
    default: return BQD_ERR_INVALID_ARG;
    }
}

}  // namespace bqd
