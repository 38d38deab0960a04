// Speculative-decoding verification in one kernel.
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析", §三: a single
// kernel (spec_decode_verify) fuses the three steps "compare the draft tokens
// -> count the accepted length -> produce the correction token".  The page
// gives no formula; the greedy reading is used:
//
//   t[b, i]       = argmax_v logits[b, i, v]     (i = 0 .. D; ties -> smallest v;
//                                                 NaN entries are never chosen;
//                                                 a row of NaNs gives -1)
//   accepted[b]   = max a in [0, D] with draft[b, i] == t[b, i] >= 0 for all i < a
//   next_token[b] = t[b, accepted[b]]            (the correction token, or the
//                                                 bonus token when all D match)
//
// Layout: logits [B, D+1, V] (fp16 or fp32), draft int32 [B, D].  One thread-
// block cluster per sequence b.  With few rows each row's vocabulary is split
// into P parts (D+1 <= 16: P = 16 / (D+1), parts of at least 4096), so that a
// sequence is read by up to 16 SMs; the cluster has C = min((D+1) P, 16) CTAs
// and rank r reduces parts r, r + C, ... (16-byte streaming loads, a
// per-thread running (value, index) best, a warp-shuffle and shared-memory
// reduction) and stores each part's best into rank 0's shared memory.  After
// the cluster barrier rank 0 combines the parts of each row in the same order,
// scans t[b, 0 ..] and writes accepted and next_token.  No global scratch, no
// atomics, no waits other than the cluster barrier.
#include <stdint.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "bqd_internal.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

constexpr int kThreadsV = 512;
constexpr int kMaxClusterV = 16;

// (value, index) order: larger value first, then smaller index; NaN values
// never win (every comparison with NaN is false)
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ float to_f(__half h) { return __half2float(h); }
__device__ __forceinline__ float to_f(float f) { return f; }

template <typename T>
__device__ __forceinline__ void take_vec(const uint4 &u, int base, float &bv, int &bi)
{
    if constexpr (sizeof(T) == 2) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(h[e]);
            if (better(f.x, base + 2 * e, bv, bi)) { bv = f.x; bi = base + 2 * e; }
            if (better(f.y, base + 2 * e + 1, bv, bi)) { bv = f.y; bi = base + 2 * e + 1; }
        }
    } else {
        const float *f = reinterpret_cast<const float *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (better(f[e], base + e, bv, bi)) { bv = f[e]; bi = base + e; }
    }
}

struct Best {
    float v;
    int i;
};

// best (value, index) of the n values at seg, reported as indices i0 + local;
// valid in thread 0 (index INT_MAX when every value is NaN)
template <typename T>
__device__ Best slice_best(const T *seg, int n, int i0, float *red_v, int *red_i)
{
    constexpr int E = 16 / sizeof(T);  // values per 16-byte load
    const int tid = threadIdx.x;
    float bv = -INFINITY;
    int bi = INT_MAX;
    // values before the first 16-byte boundary, the aligned body, the tail
    const int head = min(n, (int)(((16 - (reinterpret_cast<uintptr_t>(seg) & 15)) & 15) / sizeof(T)));
    if (tid < head) {
        const float v = to_f(seg[tid]);
        if (better(v, i0 + tid, bv, bi)) { bv = v; bi = i0 + tid; }
    }
    const int nvec = (n - head) / E;
    const uint4 *body = reinterpret_cast<const uint4 *>(seg + head);
    int q = tid;
    for (; q + 3 * kThreadsV < nvec; q += 4 * kThreadsV) {
        uint4 u[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) u[j] = __ldcs(body + q + j * kThreadsV);
#pragma unroll
        for (int j = 0; j < 4; ++j) take_vec<T>(u[j], i0 + head + (q + j * kThreadsV) * E, bv, bi);
    }
    for (; q < nvec; q += kThreadsV) take_vec<T>(__ldcs(body + q), i0 + head + q * E, bv, bi);
    for (int k = head + nvec * E + tid; k < n; k += kThreadsV) {
        const float v = to_f(seg[k]);
        if (better(v, i0 + k, bv, bi)) { bv = v; bi = i0 + k; }
    }
    // warp, then block reduction in the same order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_down_sync(0xffffffffu, bv, o);
        const int oi = __shfl_down_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        red_v[warp] = bv;
        red_i[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
        bv = lane < kThreadsV / 32 ? red_v[lane] : -INFINITY;
        bi = lane < kThreadsV / 32 ? red_i[lane] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_down_sync(0xffffffffu, bv, o);
            const int oi = __shfl_down_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
    }
    __syncthreads();  // red_* is reused by the next slice
    return Best{bv, bi};
}

template <typename T>
__global__ void __launch_bounds__(kThreadsV)
spec_verify_kernel(const T *logits, const int32_t *draft, int D, int V, int C, int P, int32_t *accepted,
                   int32_t *next_token, int32_t *argmax_out)
{
    // work item w = part w % P of row w / P (P parts of V per row); rank r of
    // the cluster takes items r, r + C, ...; their (value, index) bests are
    // gathered in rank 0's copy of these arrays
    extern __shared__ float dyn[];
    const int W = (D + 1) * P;
    float *best_v = dyn;
    int *best_i = reinterpret_cast<int *>(dyn + W);
    __shared__ float red_v[kThreadsV / 32];
    __shared__ int red_i[kThreadsV / 32];
    const int rank = C > 1 ? (int)cluster_ctarank() : 0;
    const int b = blockIdx.x / C;
    // every CTA of the cluster must have started before its shared memory is
    // written remotely: arrive now, wait after the slices are reduced
    if (C > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    for (int w = rank; w < W; w += C) {
        const int i = w / P, j = w % P;
        const int v0 = (int)((int64_t)j * V / P), v1 = (int)((int64_t)(j + 1) * V / P);
        const T *row = logits + ((size_t)b * (D + 1) + i) * (size_t)V;
        const Best bt = slice_best<T>(row + v0, v1 - v0, v0, red_v, red_i);
        if (threadIdx.x == 0) {
            best_v[w] = bt.v;
            best_i[w] = bt.i;
        }
    }
    if (C > 1) {
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (rank != 0 && threadIdx.x == 0)
            for (int w = rank; w < W; w += C) {
                uint32_t rv, ri;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rv) : "r"(smem_addr(&best_v[w])), "r"(0));
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ri) : "r"(smem_addr(&best_i[w])), "r"(0));
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(rv), "f"(best_v[w]) : "memory");
                asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ri), "r"(best_i[w]) : "memory");
            }
        cluster_sync();  // release the remote stores, acquire them in rank 0
    } else {
        __syncthreads();
    }
    if (rank == 0 && threadIdx.x == 0) {
        // t[b, i]: the best of row i's parts (same order), -1 for a row of NaNs
        auto token = [&](int i) {
            float bv = best_v[i * P];
            int bi = best_i[i * P];
            for (int j = 1; j < P; ++j)
                if (better(best_v[i * P + j], best_i[i * P + j], bv, bi)) {
                    bv = best_v[i * P + j];
                    bi = best_i[i * P + j];
                }
            return bi == INT_MAX ? -1 : bi;
        };
        int a = 0, t = token(0);
        while (a < D && t >= 0 && draft[(size_t)b * D + a] == t) {
            if (argmax_out) argmax_out[(size_t)b * (D + 1) + a] = t;
            ++a;
            t = token(a);
        }
        accepted[b] = a;
        next_token[b] = t;
        if (argmax_out) {
            argmax_out[(size_t)b * (D + 1) + a] = t;
            for (int i = a + 1; i <= D; ++i) argmax_out[(size_t)b * (D + 1) + i] = token(i);
        }
    }
}

template <typename T>
int launch_spec(const void *logits, const int32_t *draft, int64_t B, int64_t D, int64_t V, int32_t *accepted,
                int32_t *next_token, int32_t *argmax_out, cudaStream_t s)
{
    auto kern = spec_verify_kernel<T>;
    // too few rows to fill the GPU (B (D+1) below two per SM): split each
    // row's vocabulary over P CTAs of the cluster, so that a sequence is read
    // by up to 16 SMs; parts of >= 4096
    const int64_t rows = D + 1;
    int P = rows <= kMaxClusterV ? (int)(kMaxClusterV / rows) : 1;
    P = (int)std::min<int64_t>(P, std::max<int64_t>(1, V / 4096));
    if (B * rows >= 2 * (int64_t)sm_count()) P = 1;
    const int C = (int)std::min<int64_t>(rows * P, kMaxClusterV);
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * C));
    cfg.blockDim = dim3(kThreadsV);
    cfg.dynamicSmemBytes = (size_t)(D + 1) * P * (sizeof(float) + sizeof(int));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const T *>(logits), draft, (int)D, (int)V, C, P, accepted,
                              next_token, argmax_out) == cudaSuccess
               ? BQD_OK
               : BQD_ERR_CUDA;
}

}  // namespace

int launch_spec_decode_verify(const void *logits, int dtype, const int32_t *draft, int64_t B, int64_t D, int64_t V,
                              int32_t *accepted, int32_t *next_token, int32_t *argmax_out, cudaStream_t s)
{
    if (dtype == BQD_DTYPE_F16)
        return launch_spec<__half>(logits, draft, B, D, V, accepted, next_token, argmax_out, s);
    return launch_spec<float>(logits, draft, B, D, V, accepted, next_token, argmax_out, s);
}

}  // namespace bqd
