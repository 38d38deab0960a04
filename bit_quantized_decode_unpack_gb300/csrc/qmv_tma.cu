// Tensor-core decode QMV for 1-bit and 2-bit affine codes, weights streamed by
// TMA into a shared-memory ring (M <= 8 activation rows, K a multiple of 256).
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" -- §二.1
// (qmv_fast: uint32-packed codes unpacked in registers, no floating-point
// weight matrix in memory) and §二.2 (qmv_wide: one read of each weight byte
// serves all M rows; the sym variant reads no bias tensor).
//
//   y[m,n] = sum_g s[n,g] * sum_{k in g} x[m,k] q[n,k]  +  sum_g b[n,g] Sx[m,g]
//
// Unpack: one LOP3 per two codes.  It places a code q at mantissa bit p of an
// fp16 whose exponent makes its value off_p + q, off_p = 2^(10-p).  Weight
// rows are the MMA M dimension and the <= 8 x rows the N dimension
// (mma.sync m16n8k16, fp32 accumulation).  The four threads of an MMA quad
// hold codes of the SAME quantisation group, so each group's MMAs accumulate
// acc_g = sum_{k in g} x_k (off_k + q_k) on their own.  The same MMAs over
// all-zero codes give Cx_g = sum_{k in g} x_k off_k (computed once per CTA),
// and s * (acc_g - Cx_g) in fp32 is the group's scaled dot product.  A row
// whose codes in a group are all zero therefore contributes exactly zero
// (identical MMA inputs), and the scale never meets an fp16 rounding.  The
// bias term is one m16n8k8 per chunk against the group sums Sx split into an
// fp16 high part and remainder.
//
// CTA: 8 consumer warps (warp w owns two 16-row MMA tiles of weight rows, or
// one on narrow layers, for the CTA's whole K range: 256- or 128-row CTAs)
// and two producer warps, which prepare alternate ring stages (one warp alone
// bounded the pipeline with 8-column fragments).  The producers stream the
// CTA's rows chunk by chunk (256 codes per row) into
// the ring: the weight tile with one 2-D TMA copy (64- or 32-byte swizzle, so
// the quads' 32-bit reads hit 32 distinct banks), the tile's scales and
// biases once per CTA (one TMA box each when a row of them is a multiple of
// 16 bytes, else 4-byte cp.async copies by every thread), all completing on
// mbarriers.  Weights, scales and biases are requested before the
// programmatic-dependent-launch wait.
// K is split over the S CTAs of a thread-block cluster; the partial sums are
// reduce-scattered through distributed shared memory (st.async completing on
// the receiving rank's mbarrier) and added in rank order: no global scratch,
// no atomics, bit-reproducible.  Every mbarrier wait is
// bounded; on expiry the CTA stops working, drains its copies, passes its
// remaining barriers, and the expiry is counted for bqd_device_status.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "bqd_internal.cuh"
#include "qmv_codes.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

__device__ unsigned int g_qmv_tma_timeouts = 0;

constexpr int kCons = 8;                     // consumer warps
constexpr int kProd = 2;                     // producer warps: they take alternate stages
constexpr int kThreadsT = (kCons + kProd) * 32;
constexpr int kChunkT = 256;                 // codes per row per stage
constexpr int kMaxStagesT = 8;
constexpr int kMaxSplitT = 16;  // cluster sizes above 8 are the non-portable ones
constexpr size_t kSmemBudgetT = 112 * 1024;  // two CTAs per SM (with static smem and the 1 KB reserve)

struct TmaParams {
    const __half *x;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M, N, K, G, chunks, S, Cs, stages, RS, BX;
    int sc_tma;     // 1: scale / bias boxes by TMA; 0: by 4-byte cp.async copies (G % 8 != 0)
    uint32_t zero;  // always 0: keeps the magic constants opaque (in registers)
    unsigned long long wait_ns;  // limit of the pipeline waits
};

// ---- PTX wrappers local to this kernel ---------------------------------------

// pipeline waits give up after the call's limit; drain waits after a second
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    return mbar_wait_for(bar, parity, limit_ns, &g_qmv_tma_timeouts);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 4 bytes global -> shared; src_bytes 0 writes zeros and reads nothing
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// one arrival on `bar` once all of this thread's earlier cp.async copies have
// landed (counted in the barrier's expected arrivals)
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// two floats into CTA `rank`'s shared memory; the write completes 8 bytes
// of that CTA's mbarrier at the same local offset as `local_bar`
__device__ __forceinline__ void st_async_v2(uint32_t local_addr, uint32_t local_bar, uint32_t rank, float a, float b)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(ra),
                 "f"(a), "f"(b), "r"(rb)
                 : "memory");
}

// mma.sync without `volatile`, so that the compiler may schedule it freely
__device__ __forceinline__ void mma_k16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a0, a1) = fma(s, (g0, g1) - (c0, c1), (a0, a1)) on packed fp32 pairs: each
// element rounds as the scalar subtraction and fused multiply-add would
__device__ __forceinline__ void fma_sub2(float &a0, float &a1, float s, float g0, float g1, float c0, float c1)
{
    asm("{\n\t.reg .b64 g, c, d, a, ss;\n\t"
        "mov.b64 g, {%2, %3};\n\t"
        "mov.b64 c, {%4, %5};\n\t"
        "sub.rn.f32x2 d, g, c;\n\t"
        "mov.b64 ss, {%6, %6};\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "fma.rn.f32x2 a, ss, d, a;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(g0), "f"(g1), "f"(c0), "f"(c1), "f"(s));
}

__device__ __forceinline__ void mma_k8(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// shared-memory loads by 32-bit shared address
__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t a)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ uint4 ld_x16(const __half *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float h2f_lo(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w & 0xffffu))); }
__device__ __forceinline__ float h2f_hi(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w >> 16))); }

// ---- the kernel --------------------------------------------------------------------

// TPW MMA row tiles (16 rows each) per consumer warp: 2 (256-row CTAs), or 1
// (128-row CTAs, twice the CTAs of a narrow layer)
template <int TPW> constexpr int kRowsWT = 16 * TPW;          // weight rows per consumer warp
template <int TPW> constexpr int kRowsCT = kRowsWT<TPW> * kCons;  // weight rows per CTA

// One ring stage = one 256-code chunk of the CTA's rows:
//   weights [rows][CB] (TMA, swizzled) | B fragments [8][MP][4] uint4
//   | Cx [4][8] f32 | Sx as fp16 (hi, lo) [8][4]
// The scales and biases of the CTA's whole K range sit outside the ring, one
// box each: [rows][BX groups] fp16, zero past row N and group G.
// a producer's staging of one chunk of x: MP rows of 256 fp16
template <int MP>
constexpr int kXRawBytes = MP * kChunkT * 2;

template <int FMT, int GS, bool HAS_BIAS, int MP, int TPW>
struct Stage {
    static constexpr int kGPC = kChunkT / GS;
    static constexpr int kW = kRowsCT<TPW> * TF<FMT, GS>::kChunkBytes;
    static constexpr int kB = kW;
    static constexpr int kCx = kB + 8 * MP * 4 * 16;
    static constexpr int kSx = kCx + 4 * 8 * 4;
    static constexpr int kBytes = (kSx + 8 * 4 * 4 + 511) / 512 * 512;  // keeps the weight tile 512-aligned
};


template <int FMT, int GS, bool HAS_BIAS, int MP, int TPW>
__global__ void __launch_bounds__(kThreadsT, 2)
    qmv_tma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap bmap, const TmaParams p)
{
    using F = TF<FMT, GS>;
    using SL = Stage<FMT, GS, HAS_BIAS, MP, TPW>;
    constexpr int kRowsW = kRowsWT<TPW>;
    constexpr int kRowsC = kRowsCT<TPW>;
    constexpr int NR = 2 * TPW;  // rows per consumer thread: rb + 8 rr
    constexpr int GPC = SL::kGPC;
    constexpr int NPR = GS / 8;   // fp16x2 registers per (row, group)
    constexpr int MPG = GS / 16;  // MMAs per group
    constexpr uint32_t CB = F::kChunkBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStagesT], empty_bar[kMaxStagesT], sc_bar;
    __shared__ __align__(8) uint64_t red_bar;  // split K: this rank's rows of every rank's partials have landed
    __shared__ int last_it[kMaxStagesT];  // iteration whose weights a stage received last (-1: none)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int S = p.S;
    const int rank = S > 1 ? (int)cluster_ctarank() : 0;
    const int n0 = (blockIdx.x / S) * kRowsC;
    // pass blockIdx.y takes x rows 8y .. 8y+7 (M > 8 runs every pass in this one launch)
    const int M = min(8, p.M - 8 * (int)blockIdx.y);
    // B-fragment column read by thread (g, t): with 4-column fragments
    // columns 4..7 repeat 0..3; with 8 columns, columns past M repeat M - 1,
    // so the producer builds only the M real rows (outputs past M are dropped)
    const int bcol = MP == 4 ? (g & 3) : min(g, M - 1);
    const __half *xg = p.x + (size_t)(8 * blockIdx.y) * p.K;
    __half *outg = p.out + (size_t)(8 * blockIdx.y) * p.N;
    const int c_lo = rank * p.Cs;
    const int ncl = max(0, min(p.Cs, p.chunks - c_lo));
    const int NST = p.stages;

    // The next kernel in the stream may start as soon as every CTA of this one
    // runs: it prefetches its own weights and waits (griddepcontrol.wait) for
    // this grid to finish before it touches activations or outputs.
    pdl_launch_dependents();

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_a = smem_addr(smem);
    const uint32_t xraw_a = ring_a + (uint32_t)NST * SL::kBytes;  // per producer [MP][256] fp16
    const uint32_t sc_a = xraw_a + kProd * kXRawBytes<MP>;          // scales [rows][BX] fp16
    const uint32_t bi_a = sc_a + (uint32_t)(kRowsC * p.BX * 2);     // biases [rows][BX] fp16
    float *red = reinterpret_cast<float *>(smem + (size_t)NST * SL::kBytes + kProd * kXRawBytes<MP> +
                                           (size_t)kRowsC * p.BX * 2 * (HAS_BIAS ? 2 : 1));  // [S][RS][8]
    // the scale box starts at a 16-byte aligned group index
    const int g0 = c_lo * GPC, gx = g0 & ~7;

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            // producer lane 0 (expect_tx) + 32 arrivals once x is prepared
            mbar_init(smem_addr(&full_bar[s]), 33);
            mbar_init(smem_addr(&empty_bar[s]), kCons * 32);
        }
        // scale boxes: producer lane 0 (expect_tx), or every thread's copies
        mbar_init(smem_addr(&sc_bar), p.sc_tma ? 1 : kThreadsT);
        if (S > 1) {
            // rows [rank RS, rank RS + nrow) from all S ranks, ceil(M/2) float pairs a row
            const int nrow = max(0, min(p.RS, kRowsC - rank * p.RS));
            mbar_init(smem_addr(&red_bar), 1);
            mbar_arrive_expect_tx(smem_addr(&red_bar), (uint32_t)(S * nrow * ((M + 1) / 2) * 8));
        }
    }
    if (tid < kMaxStagesT) last_it[tid] = -1;
    __syncthreads();
    // split phase: every CTA of the cluster has started, with its reduction
    // barrier set up, before any distributed-shared-memory store (the matching
    // wait is before them)
    if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (!p.sc_tma && ncl > 0) {
        // rows of G fp16 that are no multiple of 16 bytes (G even, so 4-byte
        // aligned): the boxes by 4-byte copies of two groups, every thread
        // taking every kThreadsT-th pair; gx + j < G implies gx + j + 1 < G
        const int hbx = p.BX >> 1;
        for (int e = tid; e < kRowsC * hbx; e += kThreadsT) {
            const int r = e / hbx, j = 2 * (e - r * hbx);
            const bool in = n0 + r < p.N && gx + j < p.G;
            const size_t off = in ? (size_t)(n0 + r) * p.G + gx + j : 0;
            cp_async4(sc_a + (uint32_t)(4 * e), p.scales + off, in ? 4u : 0u);
            if (HAS_BIAS) cp_async4(bi_a + (uint32_t)(4 * e), p.biases + off, in ? 4u : 0u);
        }
        cp_async_arrive_noinc(smem_addr(&sc_bar));
    }
    uint32_t mg[10];
#pragma unroll
    for (int i = 0; i < 10; ++i) mg[i] = F::magic_at(i < F::kNumMagic ? i : 0) ^ p.zero;

    if (warp >= kCons) {
        // ---- producers -----------------------------------------------------------
        // Producer pw prepares the stages of chunks pw, pw + 2, ...: weights by
        // TMA, then x of the chunk turned into MMA B fragments, and Cx / Sx of
        // its groups by the same MMA sequence as the consumers (row 0: all-zero
        // codes, which unpack to exactly the magic values; row 1: ones).  With
        // M <= 4, columns 4..7 of those MMAs carry a second group.  Producer 0
        // also loads the scale (and bias) boxes.
        const int pw = warp - kCons;
        const uint32_t xr_a = xraw_a + (uint32_t)(pw * kXRawBytes<MP>);
        auto issue_weights = [&](int it, int s) {
            if (lane == 0) {
                const uint32_t bar = smem_addr(&full_bar[s]);
                mbar_arrive_expect_tx(bar, (uint32_t)SL::kW);
                tma_load_2d(ring_a + (uint32_t)s * SL::kBytes, &wmap, (c_lo + it) * (int)CB, n0, bar);
                last_it[s] = it;
            }
        };
        auto load_x = [&](int it, uint4 (&xv)[MP]) {
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                xv[m] = make_uint4(0, 0, 0, 0);
                if (m < M) xv[m] = ld_x16(xg + (size_t)m * p.K + (size_t)(c_lo + it) * kChunkT + 8 * lane);
            }
        };
        uint32_t Az[NPR];
        F::zero_group(mg, Az);
        const uint32_t one2 = 0x3C003C00u;
        // scales, biases and the weights of the first stages do not depend on
        // the previous kernel
        if (p.sc_tma && pw == 0 && lane == 0 && ncl > 0) {
            const uint32_t bx_bytes = (uint32_t)(kRowsC * p.BX * 2);
            mbar_arrive_expect_tx(smem_addr(&sc_bar), bx_bytes * (HAS_BIAS ? 2 : 1));
            tma_load_2d(sc_a, &smap, gx, n0, smem_addr(&sc_bar));
            if (HAS_BIAS) tma_load_2d(bi_a, &bmap, gx, n0, smem_addr(&sc_bar));
        }
        const int pre = min(NST, ncl);
        for (int it = pw; it < pre; it += kProd) issue_weights(it, it);
        pdl_wait();
        uint4 xv[MP];
        if (pw < ncl) load_x(pw, xv);
        for (int it = pw; it < ncl; it += kProd) {
            const int s = it % NST;
            const uint32_t par = (uint32_t)(it / NST) & 1u;
            const uint32_t st = ring_a + (uint32_t)s * SL::kBytes;
            if (it >= NST) {
                bool ok = lane == 0 ? wait_bounded(smem_addr(&empty_bar[s]), par ^ 1u, p.wait_ns) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                issue_weights(it, s);
            }
            // x of this chunk -> staging rows (zeros past M with 4-column fragments;
            // with 8 the rows past M are never read), then the next chunk's loads
#pragma unroll
            for (int m = 0; m < MP; ++m)
                if (MP == 4 || m < M)
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(xr_a + (uint32_t)(m * 512 + 16 * lane)),
                             "r"(xv[m].x), "r"(xv[m].y), "r"(xv[m].z), "r"(xv[m].w)
                             : "memory");
            if (it + kProd < ncl) load_x(it + kProd, xv);
            __syncwarp();
            // B fragments: 16 items per x row, each two 16-byte reads -> two entries
#pragma unroll
            for (int u = 0; u < MP / 2; ++u) {
                if (MP == 8 && 2 * u >= M) break;
                const int e = lane + 32 * u;
                const int i16 = e & 15, m = e >> 4;
                int base, pp0, ts;
                F::xitem(i16, base, pp0, ts);
                const uint4 vl = lds128(xr_a + (uint32_t)(m * 512 + base * 2));
                const uint4 vh = lds128(xr_a + (uint32_t)(m * 512 + (base + F::kHO) * 2));
                const uint32_t d = st + SL::kB + (uint32_t)(((pp0 * MP + m) * 4 + ts) * 16);
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(d), "r"(__byte_perm(vl.x, vh.x, 0x5410)),
                             "r"(__byte_perm(vl.x, vh.x, 0x7632)), "r"(__byte_perm(vl.y, vh.y, 0x5410)),
                             "r"(__byte_perm(vl.y, vh.y, 0x7632))
                             : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(d + MP * 4 * 16),
                             "r"(__byte_perm(vl.z, vh.z, 0x5410)), "r"(__byte_perm(vl.z, vh.z, 0x7632)),
                             "r"(__byte_perm(vl.w, vh.w, 0x5410)), "r"(__byte_perm(vl.w, vh.w, 0x7632))
                             : "memory");
            }
            __syncwarp();
            // Cx (row 0) and Sx (row 1) of the chunk's groups
            {
                constexpr int IPC = MP == 4 ? 2 : 1;
                constexpr int NCH = GPC / IPC;
                float d[NCH][4];
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) d[ch][0] = d[ch][1] = d[ch][2] = d[ch][3] = 0.f;
#pragma unroll
                for (int i = 0; i < MPG; i += 2) {
                    const uint32_t a0 = g == 0 ? Az[2 * i] : (g == 1 ? one2 : 0u);
                    const uint32_t a2 = g == 0 ? Az[2 * i + 1] : (g == 1 ? one2 : 0u);
                    const uint32_t a0n = g == 0 ? Az[2 * i + 2] : (g == 1 ? one2 : 0u);
                    const uint32_t a2n = g == 0 ? Az[2 * i + 3] : (g == 1 ? one2 : 0u);
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        const int j = ch * IPC + ((IPC == 2 && g >= 4) ? 1 : 0);
                        const int mi = j * MPG + i;
                        const uint4 b = lds128(st + SL::kB + (uint32_t)((((mi >> 1) * MP + bcol) * 4 + t) * 16));
                        mma_k16(d[ch], a0, 0u, a2, 0u, b.x, b.y);
                        mma_k16(d[ch], a0n, 0u, a2n, 0u, b.z, b.w);
                    }
                }
                if (g < 2) {
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        const int j = ch * IPC + ((IPC == 2 && t >= 2) ? 1 : 0);
                        const int col0 = IPC == 2 ? 2 * (t & 1) : 2 * t;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const float v = d[ch][h];
                            if (g == 0) {
                                asm volatile("st.shared.f32 [%0], %1;" ::"r"(st + SL::kCx + (uint32_t)((j * 8 + col0 + h) * 4)),
                                             "f"(v)
                                             : "memory");
                            } else {
                                const __half vh = __float2half_rn(v);
                                const __half vl = __float2half_rn(v - __half2float(vh));
                                const uint32_t pk = (uint32_t)__half_as_ushort(vh) | ((uint32_t)__half_as_ushort(vl) << 16);
                                const uint32_t sa = st + SL::kSx + (uint32_t)(((col0 + h) * 4 + j) * 4);
                                asm volatile("st.shared.u32 [%0], %1;" ::"r"(sa), "r"(pk) : "memory");
                                if (GPC == 2) asm volatile("st.shared.u32 [%0], %1;" ::"r"(sa + 8), "r"(0u) : "memory");
                            }
                        }
                    }
                }
                // with M <= 4 the consumers' columns 4..7 repeat columns 0..3:
                // their bias slots hold zeros
                if (MP == 4 && lane < 16)
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(st + SL::kSx + (uint32_t)((16 + lane) * 4)), "r"(0u)
                                 : "memory");
            }
            mbar_arrive(smem_addr(&full_bar[s]));
        }
        // every copy this CTA issued has landed before anyone leaves.  Only a
        // stage's last copy can still be in flight (each earlier one was
        // consumed before the stage was refilled), and each issued stage was
        // also prepared, so its barrier can complete: once both producers have
        // stopped issuing, each waits for the stages it filled last
        if (!p.sc_tma) cp_async_wait_all();  // this thread's scale copies
        asm volatile("bar.sync 1, %0;" ::"n"(kProd * 32) : "memory");
        if (lane == 0) {
            for (int s = 0; s < NST; ++s) {
                const int li = last_it[s];
                if (li >= 0 && li % kProd == pw)
                    wait_bounded(smem_addr(&full_bar[s]), (uint32_t)(li / NST) & 1u, kDrainWaitNs);
            }
            if (pw == 0 && ncl > 0) wait_bounded(smem_addr(&sc_bar), 0, kDrainWaitNs);
        }
        __syncwarp();
        if (S > 1) {
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
        }
        return;
    }

    // ---- consumers: warp w owns rows 32w .. 32w+31 (two MMA row tiles) -------------
    float acc[TPW][4];
#pragma unroll
    for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[tl][q] = 0.f;
    const int rb = warp * kRowsW + g;  // rows rb, rb+8 (tile 0), rb+16, rb+24 (tile 1)
    const int jb = t & (GPC - 1);      // bias slot t: group t (gs=64), group t&1 for t < 2 (gs=128)
    uint32_t woff[F::kNW];
#pragma unroll
    for (int v = 0; v < F::kNW; ++v) woff[v] = F::word_off(rb, v, t);  // rows +8/16/24 share its swizzle
    // scales / biases of row rb, group g0 - gx + GPC*it (+ jb for the bias slot)
    const uint32_t R8S = (uint32_t)(8 * p.BX * 2);
    uint32_t sq = sc_a + (uint32_t)((rb * p.BX + g0 - gx) * 2);
    uint32_t bqb = bi_a + (uint32_t)((rb * p.BX + g0 - gx + jb) * 2);
    const uint32_t bqo = (uint32_t)(SL::kB + ((bcol * 4) + t) * 16);
    const uint32_t cxo = (uint32_t)(SL::kCx + 8 * t);
    const uint32_t sxo = (uint32_t)(SL::kSx + (g * 4 + t) * 4);
    // words of group j that a thread unpacks (per row): GS/64 for 2-bit, one for 1-bit
    constexpr int WPG = FMT == BQD_FMT_AFFINE2 ? GS / 64 : 1;
    uint32_t st_a = ring_a;
    int s = 0;
    uint32_t par = 0;
    const bool sc_ok = ncl == 0 || wait_bounded(smem_addr(&sc_bar), 0, p.wait_ns);
    // the box barrier completes only once every thread's scale copies have
    // landed; after an expired wait this thread's own may still be in flight
    if (!sc_ok) cp_async_wait_all();
    for (int it = 0; it < ncl && sc_ok; ++it) {
        if (!wait_bounded(smem_addr(&full_bar[s]), par, p.wait_ns)) break;
        // scales of the four rows for the chunk's groups
        uint32_t sw[NR][GPC / 2];
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) {
            if constexpr (GPC == 4) {
                const uint2 a = lds64(sq + rr * R8S);
                sw[rr][0] = a.x;
                sw[rr][GPC / 2 - 1] = a.y;
            } else {
                sw[rr][0] = lds32(sq + rr * R8S);
            }
        }
        // bias term first, straight into the accumulators
        {
            uint16_t bb[NR];
#pragma unroll
            for (int rr = 0; rr < NR; ++rr) {
                if constexpr (HAS_BIAS) {
                    bb[rr] = lds16(bqb + rr * R8S);
                } else {
                    const uint32_t x0 = (jb >> 1) ? sw[rr][GPC / 2 - 1] : sw[rr][0];
                    bb[rr] = __half_as_ushort(sym_bias(__ushort_as_half((uint16_t)(x0 >> (16 * (jb & 1)))), p.ratio));
                }
                if (GPC == 2 && t >= 2) bb[rr] = 0;
            }
            const uint32_t sxv = lds32(st_a + sxo);
#pragma unroll
            for (int tl = 0; tl < TPW; ++tl) mma_k8(acc[tl], dup_half(bb[2 * tl]), dup_half(bb[2 * tl + 1]), sxv);
        }
        const uint32_t bq = st_a + bqo;
#pragma unroll
        for (int j = 0; j < GPC; ++j) {
            // this group's words of the thread's rows, read when needed
            uint32_t w[NR][F::kNW];
#pragma unroll
            for (int rr = 0; rr < NR; ++rr)
#pragma unroll
                for (int v = 0; v < WPG; ++v) {
                    const int idx = j * WPG + v;
                    w[rr][idx] = lds32(st_a + woff[idx] + rr * 8 * CB);
                }
            float ag[TPW][4];
#pragma unroll
            for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
                for (int q = 0; q < 4; ++q) ag[tl][q] = 0.f;
#pragma unroll
            for (int tl = 0; tl < TPW; ++tl) {
                uint32_t A0[NPR], A1[NPR];
                F::unpack_group(w[2 * tl], j, t, mg, A0);
                F::unpack_group(w[2 * tl + 1], j, t, mg, A1);
#pragma unroll
                for (int i = 0; i < MPG; i += 2) {
                    const int mi = j * MPG + i;
                    const uint4 b = lds128(bq + (uint32_t)((mi >> 1) * MP * 4 * 16));
                    mma_k16(ag[tl], A0[2 * i], A1[2 * i], A0[2 * i + 1], A1[2 * i + 1], b.x, b.y);
                    mma_k16(ag[tl], A0[2 * i + 2], A1[2 * i + 2], A0[2 * i + 3], A1[2 * i + 3], b.z, b.w);
                }
            }
            const uint2 cxv = lds64(st_a + cxo + (uint32_t)(j * 32));
            const float cx0 = __uint_as_float(cxv.x), cx1 = __uint_as_float(cxv.y);
#pragma unroll
            for (int tl = 0; tl < TPW; ++tl) {
                const float sa = (j & 1) ? h2f_hi(sw[2 * tl][j >> 1]) : h2f_lo(sw[2 * tl][j >> 1]);
                const float sb = (j & 1) ? h2f_hi(sw[2 * tl + 1][j >> 1]) : h2f_lo(sw[2 * tl + 1][j >> 1]);
                fma_sub2(acc[tl][0], acc[tl][1], sa, ag[tl][0], ag[tl][1], cx0, cx1);
                fma_sub2(acc[tl][2], acc[tl][3], sb, ag[tl][2], ag[tl][3], cx0, cx1);
            }
        }
        mbar_arrive(smem_addr(&empty_bar[s]));
        sq += GPC * 2;
        bqb += GPC * 2;
        st_a += SL::kBytes;
        if (++s == NST) {
            s = 0;
            par ^= 1u;
            st_a = ring_a;
        }
    }

    // ---- results -------------------------------------------------------------------
    // value (tile tl, q) is row rb + 16 tl + 8 (q >> 1), column 2t + (q & 1)
    if (S == 1) {
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = n0 + rb + 16 * tl + 8 * (q >> 1), m = 2 * t + (q & 1);
                if (n < p.N && m < M) outg[(size_t)m * p.N + n] = __float2half_rn(acc[tl][q]);
            }
        return;
    }
    // reduce-scatter through distributed shared memory: rank q adds rows
    // [q RS, (q+1) RS) of every rank's partials, in rank order.  Each rank
    // sends its column pairs below M with st.async, which completes bytes of
    // the receiving rank's red_bar; a rank reads its rows once all have
    // landed.  The cluster barrier split around the reduction keeps every CTA
    // resident until every rank has received all of its rows.
    const int RS = p.RS;
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (2 * t < M) {
        const uint32_t rbar = smem_addr(&red_bar);
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = rb + 16 * tl + 8 * h;
                const int q = row / RS;
                st_async_v2(smem_addr(red + ((size_t)rank * RS + (row - q * RS)) * 8 + 2 * t), rbar, (uint32_t)q,
                            acc[tl][2 * h], acc[tl][2 * h + 1]);
            }
    }
    // every rank sends all of its rows whatever its own waits did, so this
    // wait keeps the long limit of the drains
    wait_bounded(smem_addr(&red_bar), 0, kDrainWaitNs);
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const int row0 = rank * RS;
    const int nrow = max(0, min(RS, kRowsC - row0));
    for (int e = tid; e < nrow * M; e += kCons * 32) {
        const int lr = e / M, m = e % M;
        float v = 0.f;
        for (int k = 0; k < S; ++k) v += red[((size_t)k * RS + lr) * 8 + m];
        const int n = n0 + row0 + lr;
        if (n < p.N) outg[(size_t)m * p.N + n] = __float2half_rn(v);
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// ---- host side -------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

struct TPlan {
    int S, Cs, stages, R, RS, BX;
    size_t smem;
};

template <int FMT, int GS, bool HAS_BIAS, int MP, int TPW>
size_t tma_smem(int S, int stages, int RS, int BX)
{
    return 1024 + (size_t)stages * Stage<FMT, GS, HAS_BIAS, MP, TPW>::kBytes + kProd * kXRawBytes<MP> +
           (size_t)kRowsCT<TPW> * BX * 2 * (HAS_BIAS ? 2 : 1) + (size_t)S * RS * 8 * 4;
}

template <int FMT, int GS, bool HAS_BIAS, int MP, int TPW>
int cluster_slots_t(int S, size_t smem)
{
    struct Entry { int dev, S; size_t smem; int slots; };
    static Entry cache[128];
    static int n = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].dev == dev && cache[i].S == S && cache[i].smem == smem) return cache[i].slots;
    auto kern = qmv_tma_kernel<FMT, GS, HAS_BIAS, MP, TPW>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudgetT);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(kThreadsT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = S;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int slots = 0;
    if (cudaOccupancyMaxActiveClusters(&slots, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        slots = 0;
    }
    if (n < 128) cache[n++] = Entry{dev, S, smem, slots};
    return slots;
}

// P passes of x rows run side by side in one launch (grid rows)
template <int FMT, int GS, bool HAS_BIAS, int MP, int TPW>
bool plan_t(int N, int chunks, int P, TPlan &best)
{
    constexpr int GPC = kChunkT / GS;
    constexpr int kRowsC = kRowsCT<TPW>;
    const int R = (N + kRowsC - 1) / kRowsC;
    const int sms = sm_count();
    const size_t stage = Stage<FMT, GS, HAS_BIAS, MP, TPW>::kBytes;
    double best_cost = 1e30;
    bool found = false;
    for (int S = 1; S <= kMaxSplitT && S <= chunks; ++S) {
        const int Cs = (chunks + S - 1) / S;
        if ((S - 1) * Cs >= chunks) continue;
        const int RS = (kRowsC + S - 1) / S;
        // every rank owns rows of the reduction (128 rows over 14 ranks would
        // leave the last one none)
        if ((S - 1) * RS >= kRowsC) continue;
        // scale box: the rank's groups from the 16-byte aligned group below its first
        int maxoff = 0;
        for (int r = 0; r < S; ++r) maxoff = std::max(maxoff, (r * Cs * GPC) & 7);
        const int BX = (Cs * GPC + maxoff + 7) / 8 * 8;
        if (BX > 256) continue;
        const size_t fixed = tma_smem<FMT, GS, HAS_BIAS, MP, TPW>(S, 0, RS, BX);
        if (fixed + stage > kSmemBudgetT) continue;
        int st = (int)((kSmemBudgetT - fixed) / stage);
        st = st > kMaxStagesT ? kMaxStagesT : st;
        st = st > Cs ? Cs : st;
        if (st < 2 && Cs > 1) continue;
        const size_t sm = tma_smem<FMT, GS, HAS_BIAS, MP, TPW>(S, st, RS, BX);
        const int slots = S == 1 ? 2 * sms : cluster_slots_t<FMT, GS, HAS_BIAS, MP, TPW>(S, sm);
        if (slots <= 0) continue;
        const int waves = (R * P + slots - 1) / slots;
        // time ~ waves x (chunks per CTA + first-stage latency and reduction, ~2 chunks)
        const double cost = (double)waves * (Cs + 2) + 0.1 * S;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = TPlan{S, Cs, st, R, RS, BX, sm};
            found = true;
        }
    }
    return found;
}

// 2-D tensor map of a row-major [rows][cols] fp16 array, box {box_cols, box_rows}
bool encode_f16(CUtensorMap &map, const __half *base, int64_t cols, int64_t rows, int box_cols, int box_rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int GS, bool HAS_BIAS, int MP, int TPW>
int launch_t(const TmaParams &p0, const CUtensorMap &map, int chunks, cudaStream_t s)
{
    TPlan pl;
    const int P = (p0.M + 7) / 8;
    if (!plan_t<FMT, GS, HAS_BIAS, MP, TPW>(p0.N, chunks, P, pl)) return BQD_ERR_UNSUPPORTED;
    TmaParams p = p0;
    p.S = pl.S;
    p.Cs = pl.Cs;
    p.stages = pl.stages;
    p.RS = pl.RS;
    p.BX = pl.BX;
    CUtensorMap smap{}, bmap{};  // unused (zero) when the boxes are copied by cp.async
    if (p.sc_tma) {
        if (!encode_f16(smap, p.scales, p.G, p.N, pl.BX, kRowsCT<TPW>)) return BQD_ERR_CUDA;
        bmap = smap;
        if (HAS_BIAS && !encode_f16(bmap, p.biases, p.G, p.N, pl.BX, kRowsCT<TPW>)) return BQD_ERR_CUDA;
    }
    if (opt_debug_plan())
        fprintf(stderr,
                "bqd tma plan: N=%d K=%d M=%d gs=%d -> rows=%d S=%d Cs=%d stages=%d R=%d BX=%d grid=%dx%d smem=%zu\n",
                p.N, p.K, p.M, GS, kRowsCT<TPW>, pl.S, pl.Cs, pl.stages, pl.R, pl.BX, pl.R * pl.S, P, pl.smem);
    auto kern = qmv_tma_kernel<FMT, GS, HAS_BIAS, MP, TPW>;
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudgetT) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.R * pl.S, P);
    cfg.blockDim = dim3(kThreadsT);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (pl.S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pl.S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, map, smap, bmap, p) == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
}

template <int FMT, int GS, int TPW>
int launch_fmt_gs(const TmaParams &p, const CUtensorMap &map, int chunks, bool has_bias, int MP, cudaStream_t s)
{
    if (MP == 4)
        return has_bias ? launch_t<FMT, GS, true, 4, TPW>(p, map, chunks, s)
                        : launch_t<FMT, GS, false, 4, TPW>(p, map, chunks, s);
    return has_bias ? launch_t<FMT, GS, true, 8, TPW>(p, map, chunks, s)
                    : launch_t<FMT, GS, false, 8, TPW>(p, map, chunks, s);
}

template <int FMT, int GS>
int launch_fmt_gs(const TmaParams &p, const CUtensorMap &map, int chunks, bool has_bias, int MP, int tpw,
                  cudaStream_t s)
{
    return tpw == 1 ? launch_fmt_gs<FMT, GS, 1>(p, map, chunks, has_bias, MP, s)
                    : launch_fmt_gs<FMT, GS, 2>(p, map, chunks, has_bias, MP, s);
}

}  // namespace

int take_qmv_tma_timeouts(unsigned int *count)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmv_tma_timeouts, sizeof(v)) != cudaSuccess) return BQD_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_qmv_tma_timeouts, &zero, sizeof(zero)) != cudaSuccess) return BQD_ERR_CUDA;
    *count = v;
    return BQD_OK;
}

int launch_qmv_tma(const QmvArgs &a, cudaStream_t s)
{
    if (a.fmt != BQD_FMT_AFFINE1 && a.fmt != BQD_FMT_AFFINE2) return BQD_ERR_UNSUPPORTED;
    // whole 256-code chunks; the weight tile's TMA box needs a 16-byte aligned
    // base and rows.  Scales / biases: TMA boxes when their rows (G fp16) and
    // bases are 16-byte aligned, else 4-byte copies (even G, 4-byte bases)
    if (a.K % kChunkT != 0 || a.row_bytes % 16 != 0) return BQD_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(a.w) & 15) || (reinterpret_cast<uintptr_t>(a.x) & 15)) return BQD_ERR_UNSUPPORTED;
    auto sc_align = [&](uintptr_t m) {
        return !(reinterpret_cast<uintptr_t>(a.scales) & m) && !(a.biases && (reinterpret_cast<uintptr_t>(a.biases) & m));
    };
    const bool sc_tma = a.G % 8 == 0 && sc_align(15);
    if (!sc_tma && (a.G % 2 != 0 || !sc_align(3))) return BQD_ERR_UNSUPPORTED;
    if (a.K > (int64_t)1 << 28 || a.N > (int64_t)1 << 28) return BQD_ERR_UNSUPPORTED;
    auto enc = encode_fn();
    if (!enc) return BQD_ERR_UNSUPPORTED;

    const bool b64 = a.fmt == BQD_FMT_AFFINE2;
    // narrow layers (at most eight 256-row blocks): 128-row CTAs, one 16-row
    // tile per consumer warp, so that twice the CTAs share the work and a
    // warp's work per stage halves
    const int tpw = a.N <= 2048 ? 1 : 2;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)a.row_bytes, (cuuint64_t)a.N};
    cuuint64_t strides[1] = {(cuuint64_t)a.row_bytes};
    cuuint32_t box[2] = {b64 ? 64u : 32u, (cuuint32_t)(16 * tpw * kCons)};
    cuuint32_t estr[2] = {1, 1};
    CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.w), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, b64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return BQD_ERR_CUDA;

    TmaParams p;
    p.scales = a.scales; p.biases = a.biases; p.ratio = a.ratio;
    p.N = (int)a.N; p.K = (int)a.K; p.G = (int)a.G;
    p.sc_tma = sc_tma ? 1 : 0;
    p.chunks = (int)(a.K / kChunkT);
    p.zero = 0;
    p.wait_ns = (unsigned long long)opt_wait_ns();
    p.S = p.Cs = p.stages = p.RS = 0;
    const bool hb = a.biases != nullptr;
    // M <= 8: one pass with 4 or 8 B-fragment columns; larger M: passes of 8
    // x rows, all in one launch (grid row y = rows 8y .. 8y+7), so that the
    // fixed cost of a call is paid once and later passes find the weights in L2
    if (a.M > (int64_t)8 * 65535) return BQD_ERR_UNSUPPORTED;
    const int MP = a.M <= 4 ? 4 : 8;
    p.M = (int)a.M;
    p.x = a.x;
    p.out = a.out;
    if (b64)
        return a.gs == 64 ? launch_fmt_gs<BQD_FMT_AFFINE2, 64>(p, map, p.chunks, hb, MP, tpw, s)
                          : launch_fmt_gs<BQD_FMT_AFFINE2, 128>(p, map, p.chunks, hb, MP, tpw, s);
    return a.gs == 64 ? launch_fmt_gs<BQD_FMT_AFFINE1, 64>(p, map, p.chunks, hb, MP, tpw, s)
                      : launch_fmt_gs<BQD_FMT_AFFINE1, 128>(p, map, p.chunks, hb, MP, tpw, s);
}

}  // namespace bqd
