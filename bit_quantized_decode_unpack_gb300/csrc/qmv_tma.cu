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
// CTA: 8 consumer warps (warp w owns weight rows n0+16w .. n0+16w+15 for the
// CTA's whole K range) and one producer warp.  The producer streams the
// CTA's 128 rows chunk by chunk (256 codes per row) into a ring of stages:
// the weight tile with one 2-D TMA copy (64- or 32-byte swizzle, so the
// quads' 32-bit reads hit 32 distinct banks), the tile's scales and biases
// with cp.async, all completing on the stage's mbarrier.  Weights, scales
// and biases are requested before the programmatic-dependent-launch wait.
// K is split over the S CTAs of a thread-block cluster; the partial sums are
// added in a fixed order through distributed shared memory into rank 0: no
// global scratch, no atomics, bit-reproducible.  Every mbarrier wait is
// bounded; on expiry the CTA stops working, drains its copies, passes its
// remaining barriers, and the expiry is counted for bqd_device_status.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "bqd_internal.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

__device__ unsigned int g_qmv_tma_timeouts = 0;

constexpr int kCons = 8;                     // consumer warps
constexpr int kThreadsT = (kCons + 1) * 32;  // + one producer warp
constexpr int kRowsT = 16 * kCons;           // weight rows per CTA
constexpr int kChunkT = 256;                 // codes per row per stage
constexpr int kMaxStagesT = 8;
constexpr int kMaxSplitT = 8;
constexpr size_t kSmemBudgetT = 112 * 1024;  // two CTAs per SM (with static smem and the 1 KB reserve)

struct TmaParams {
    const __half *x;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M, N, K, G, chunks, S, Cs, stages;
    uint32_t ring_bytes;
    uint32_t zero;  // always 0: keeps the magic constants opaque (in registers)
};

// ---- PTX wrappers local to this kernel ---------------------------------------

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitSpins; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicAdd(&g_qmv_tma_timeouts, 1u);
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// cp.async of BYTES (4 or 8) bytes; src_bytes = 0 writes zeros and reads nothing
template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(BYTES), "r"(src_bytes)
                 : "memory");
}

// arrive on `bar` once this thread's earlier cp.async copies have landed
// (the barrier's expected count includes this arrival)
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCons * 32) : "memory"); }

__device__ __forceinline__ void st_cluster_v2(uint32_t local_addr, uint32_t rank, float a, float b)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(a), "f"(b) : "memory");
}

// ---- format traits -------------------------------------------------------------
//
// Per chunk a thread reads kNW words of each of its two rows (g and g+8 of its
// warp's tile) from the stage.  Per (row, group) it turns them into GS/8
// fp16x2 registers A[i] (pair i = two codes 16 bits apart in one word); MMA i
// of the group takes A[2i], A[2i+1] of rows g and g+8.  The B fragment of an
// even MMA index 2pp (thread slot t) holds x at (k0+q, k0+q+HO | k0+q+1,
// k0+q+HO+1), the next MMA the same at q+2.  x is staged in 16 "items" per
// (chunk, x row): item i covers x[base .. base+7] and x[base+HO .. base+HO+7]
// and fills the entries (pp0 + h, slot tslot), h = 0, 1.

template <int FMT, int GS> struct TF;

// 2-bit: 16 codes per word, pair i = (code i, code i+8).  A 256-code chunk
// is 64 bytes per row = four 16-byte pieces of 64 codes; thread t reads word
// t of each piece (a group is GS/64 pieces).  Codes 0..4 are read from w at
// mantissa bits 0,2,4,6,8 (offsets 1024 .. 4), codes 5..7 from w >> 6 at
// bits 4,6,8: one shift per word.
template <int GS> struct TF<BQD_FMT_AFFINE2, GS> {
    static constexpr int kChunkBytes = 64;
    static constexpr int kHO = 8;
    static constexpr int kNumMagic = 5;
    static constexpr int kNW = 4;
    __host__ __device__ static constexpr uint32_t magic_at(int i) { return magic(2 * i); }

    // 64-byte rows, 64-byte swizzle: piece P of row r sits at piece P ^ ((r >> 1) & 3)
    __device__ static __forceinline__ uint32_t word_off(int r, int P, int t)
    {
        return (uint32_t)(r * 64 + ((P ^ ((r >> 1) & 3)) << 4) + 4 * t);
    }
    __device__ static __forceinline__ void unpack_word(uint32_t w, const uint32_t (&mg)[10], uint32_t *A)
    {
        const uint32_t ub = w >> 6;
        A[0] = and_or<0x00030003u << 0>(w, mg[0]);
        A[1] = and_or<0x00030003u << 2>(w, mg[1]);
        A[2] = and_or<0x00030003u << 4>(w, mg[2]);
        A[3] = and_or<0x00030003u << 6>(w, mg[3]);
        A[4] = and_or<0x00030003u << 8>(w, mg[4]);
        A[5] = and_or<0x00030003u << 4>(ub, mg[2]);
        A[6] = and_or<0x00030003u << 6>(ub, mg[3]);
        A[7] = and_or<0x00030003u << 8>(ub, mg[4]);
    }
    __device__ static __forceinline__ void unpack_group(const uint32_t (&w)[kNW], int j, int t,
                                                        const uint32_t (&mg)[10], uint32_t (&A)[GS / 8])
    {
#pragma unroll
        for (int v = 0; v < GS / 64; ++v) unpack_word(w[j * (GS / 64) + v], mg, &A[8 * v]);
    }
    __device__ static __forceinline__ void zero_group(const uint32_t (&mg)[10], uint32_t (&A)[GS / 8])
    {
#pragma unroll
        for (int v = 0; v < GS / 64; ++v) unpack_word(0u, mg, &A[8 * v]);
    }
    __device__ static __forceinline__ void xitem(int i, int &base, int &pp0, int &tslot)
    {
        const int P = i >> 2;
        tslot = i & 3;
        base = 64 * P + 16 * tslot;
        pp0 = 2 * P;
    }
};

// 1-bit: 32 codes per word, pair i = (code i, code i+16).  A chunk is 32
// bytes per row = 8 words.  Codes sit at mantissa bits 0..9 (offsets 1024 ..
// 2), one shift per word.
//   gs=64 : a group is 2 words; threads 2h, 2h+1 share word h, thread t
//           takes codes 8(t&1) .. 8(t&1)+7 (and +16), from w >> 8(t&1).
//   gs=128: a group is 4 words; thread t takes word t: codes 0..9 from w,
//           codes 10..15 from w >> 10.
template <int GS> struct TF<BQD_FMT_AFFINE1, GS> {
    static constexpr int kChunkBytes = 32;
    static constexpr int kHO = 16;
    static constexpr int kNumMagic = 10;
    static constexpr int kNW = 256 / GS;  // one word per group
    __host__ __device__ static constexpr uint32_t magic_at(int i) { return magic(i); }

    // 32-byte rows, 32-byte swizzle: piece P of row r sits at piece P ^ ((r >> 2) & 1)
    __device__ static __forceinline__ uint32_t word_off(int r, int j, int t)
    {
        const int W = GS == 64 ? 2 * j + (t >> 1) : 4 * j + t;
        return (uint32_t)(r * 32 + (((W >> 2) ^ ((r >> 2) & 1)) << 4) + 4 * (W & 3));
    }
    // A[i] = code i of u at bit i (and its partner at bit 16+i) over magic(i), i < NP
    template <int NP, int I = 0>
    __device__ static __forceinline__ void unpack_from(uint32_t u, const uint32_t (&mg)[10], uint32_t *A)
    {
        if constexpr (I < NP) {
            A[I] = and_or<(0x00010001u << I)>(u, mg[I]);
            unpack_from<NP, I + 1>(u, mg, A);
        }
    }
    __device__ static __forceinline__ void unpack_group(const uint32_t (&w)[kNW], int j, int t,
                                                        const uint32_t (&mg)[10], uint32_t (&A)[GS / 8])
    {
        if constexpr (GS == 64) {
            unpack_from<8>(w[j] >> (8 * (t & 1)), mg, &A[0]);
        } else {
            unpack_from<10>(w[j], mg, &A[0]);
            unpack_from<6>(w[j] >> 10, mg, &A[10]);
        }
    }
    __device__ static __forceinline__ void zero_group(const uint32_t (&mg)[10], uint32_t (&A)[GS / 8])
    {
        if constexpr (GS == 64) {
            unpack_from<8>(0u, mg, &A[0]);
        } else {
            unpack_from<10>(0u, mg, &A[0]);
            unpack_from<6>(0u, mg, &A[10]);
        }
    }
    __device__ static __forceinline__ void xitem(int i, int &base, int &pp0, int &tslot)
    {
        if constexpr (GS == 64) {
            const int j = i >> 2;
            tslot = i & 3;
            base = 32 * (2 * j + (tslot >> 1)) + 8 * (tslot & 1);
            pp0 = 2 * j;
        } else {
            const int j = i >> 3, u = i & 1;
            tslot = (i >> 1) & 3;
            base = 32 * (4 * j + tslot) + 8 * u;
            pp0 = 4 * j + 2 * u;
        }
    }
};

// mma.sync without `volatile`, so that the compiler may schedule it freely
__device__ __forceinline__ void mma_k16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

template <int FMT, int GS>
struct Layout {
    static constexpr int kW = kRowsT * TF<FMT, GS>::kChunkBytes;  // weight tile bytes
    static constexpr int kGPC = kChunkT / GS;                      // groups per chunk
    static constexpr int kS = kRowsT * kGPC * 2;                   // scale (or bias) tile bytes
    __host__ __device__ static constexpr int stage(bool bias) { return kW + kS * (bias ? 2 : 1); }
};

template <int FMT, int GS, bool HAS_BIAS, int MP>
__global__ void __launch_bounds__(kThreadsT, 2) qmv_tma_kernel(const __grid_constant__ CUtensorMap wmap, const TmaParams p)
{
    using F = TF<FMT, GS>;
    using L = Layout<FMT, GS>;
    constexpr int GPC = L::kGPC;
    constexpr int NPR = GS / 8;   // fp16x2 registers per (row, group)
    constexpr int MPG = GS / 16;  // MMAs per group
    constexpr int STAGE = L::stage(HAS_BIAS);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStagesT], empty_bar[kMaxStagesT];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.S;
    const int rank = S > 1 ? (int)cluster_ctarank() : 0;
    const int n0 = (blockIdx.x / S) * kRowsT;
    const int c_lo = rank * p.Cs;
    const int ncl = max(0, min(p.Cs, p.chunks - c_lo));
    const int NST = p.stages;

    // The next kernel in the stream may start as soon as every CTA of this one
    // runs: it prefetches its own weights and waits (griddepcontrol.wait) for
    // this grid to finish before it touches activations or outputs.
    pdl_launch_dependents();
    // split phase: every CTA of the cluster has started before any
    // distributed-shared-memory store (the matching wait is before them)
    if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint4 *Bs = reinterpret_cast<uint4 *>(smem + p.ring_bytes);            // [Cs][8][MP][4]
    float *Cx = reinterpret_cast<float *>(Bs + (size_t)p.Cs * 8 * MP * 4);  // [Cs][4][8]
    uint32_t *SxB = reinterpret_cast<uint32_t *>(Cx + (size_t)p.Cs * 32);  // [Cs][8][4]
    float *red = reinterpret_cast<float *>(SxB + (size_t)p.Cs * 32);       // [S-1][128][8], rank 0's is used

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 33);  // producer lane 0 (expect_tx) + 32 cp.async arrivals
            mbar_init(smem_addr(&empty_bar[s]), kCons * 32);
        }
    }
    __syncthreads();

    if (warp == kCons) {
        // ---- producer: weights by TMA, scales/biases by cp.async -----------------
        // The first NST stages need no free slot and are requested at once (they
        // do not depend on the previous kernel); later ones wait for a slot
        // after griddepcontrol.wait, so no wait spins while an earlier kernel runs.
        int issued = 0, s = 0;
        uint32_t par = 0;
        for (int it = 0; it < ncl; ++it) {
            if (it == NST) pdl_wait();
            if (it >= NST) {
                bool ok = lane == 0 ? wait_bounded(smem_addr(&empty_bar[s]), par ^ 1u) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            const uint32_t bar = smem_addr(&full_bar[s]);
            uint8_t *st = ring + (size_t)s * STAGE;
            const int c = c_lo + it;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, (uint32_t)L::kW);
                tma_load_2d(smem_addr(st), &wmap, c * F::kChunkBytes, n0, bar);
            }
#pragma unroll
            for (int i = 0; i < kRowsT / 32; ++i) {
                const int r = lane + 32 * i;
                const int n = n0 + r;
                const bool ok = n < p.N;
                const long long off = (long long)(ok ? n : 0) * p.G + (long long)c * GPC;
                cp_async<GPC * 2>(smem_addr(st + L::kW + r * GPC * 2), p.scales + off, ok ? GPC * 2 : 0);
                if (HAS_BIAS)
                    cp_async<GPC * 2>(smem_addr(st + L::kW + L::kS + r * GPC * 2), p.biases + off, ok ? GPC * 2 : 0);
            }
            cp_async_arrive_noinc(bar);
            issued = it + 1;
            if (++s == NST) {
                s = 0;
                par ^= 1u;
            }
        }
        // every copy this CTA issued has landed before anyone leaves
        if (lane == 0)
            for (int it = max(0, issued - NST); it < issued; ++it)
                wait_bounded(smem_addr(&full_bar[it % NST]), (it / NST) & 1);
        __syncwarp();
        if (S > 1) {
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        }
        return;
    }

    // ---- consumers ---------------------------------------------------------------
    const int g = lane >> 2, t = lane & 3;
    pdl_wait();
    // x -> B fragments: 16 items per (chunk, x row), four items per thread in
    // flight, each two 16-byte loads filling two entries
    {
        const int items = ncl * MP * 16;
        for (int e0 = tid; e0 < items; e0 += 4 * kCons * 32) {
            uint4 vl[4], vh[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * kCons * 32;
                const int i16 = e & 15, m = (e >> 4) % MP, c = e / (16 * MP);
                int base, pp0, ts;
                F::xitem(i16, base, pp0, ts);
                vl[u] = vh[u] = make_uint4(0, 0, 0, 0);
                if (e < items && m < p.M) {
                    const __half *xr = p.x + (size_t)m * p.K + (size_t)(c_lo + c) * kChunkT + base;
                    vl[u] = ld_x16(xr);
                    vh[u] = ld_x16(xr + F::kHO);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * kCons * 32;
                if (e >= items) continue;
                const int i16 = e & 15, m = (e >> 4) % MP, c = e / (16 * MP);
                int base, pp0, ts;
                F::xitem(i16, base, pp0, ts);
                uint4 *d = Bs + (((size_t)c * 8 + pp0) * MP + m) * 4 + ts;
                d[0] = make_uint4(__byte_perm(vl[u].x, vh[u].x, 0x5410), __byte_perm(vl[u].x, vh[u].x, 0x7632),
                                  __byte_perm(vl[u].y, vh[u].y, 0x5410), __byte_perm(vl[u].y, vh[u].y, 0x7632));
                d[MP * 4] = make_uint4(__byte_perm(vl[u].z, vh[u].z, 0x5410), __byte_perm(vl[u].z, vh[u].z, 0x7632),
                                       __byte_perm(vl[u].w, vh[u].w, 0x5410), __byte_perm(vl[u].w, vh[u].w, 0x7632));
            }
        }
    }
    consumers_sync();
    uint32_t mg[10];
#pragma unroll
    for (int i = 0; i < 10; ++i) mg[i] = F::magic_at(i < F::kNumMagic ? i : 0) ^ p.zero;
    const uint32_t bs_a = smem_addr(Bs), cx_a = smem_addr(Cx), sx_a = smem_addr(SxB);
    // Cx (the offsets' dot products, MMA row 0) and Sx (group sums, row 1) of
    // each (chunk, group), by the same MMA sequence as the main loop: row 0 of
    // A holds all-zero codes, i.e. exactly the magic values.  With M <= 4 the
    // columns 4..7 carry a second (chunk, group).
    {
        constexpr int IPC = MP == 4 ? 2 : 1;
        uint32_t Az[NPR];
        F::zero_group(mg, Az);
        const uint32_t one2 = 0x3C003C00u;
        const int items = ncl * GPC;
        for (int ch = warp; ch * IPC < items; ch += kCons) {
            int it_l = ch * IPC + ((IPC == 2 && g >= 4) ? 1 : 0);
            if (it_l >= items) it_l = ch * IPC;
            const int c = it_l / GPC, j = it_l % GPC;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t bq = bs_a + (uint32_t)((((c * 8) * MP + (g & (MP - 1))) * 4 + t) * 16);
#pragma unroll
            for (int i = 0; i < MPG; i += 2) {
                const int mi = j * MPG + i;
                const uint4 b = lds128(bq + (uint32_t)((mi >> 1) * MP * 4 * 16));
                const uint32_t a0 = g == 0 ? Az[2 * i] : (g == 1 ? one2 : 0u);
                const uint32_t a2 = g == 0 ? Az[2 * i + 1] : (g == 1 ? one2 : 0u);
                const uint32_t a0n = g == 0 ? Az[2 * i + 2] : (g == 1 ? one2 : 0u);
                const uint32_t a2n = g == 0 ? Az[2 * i + 3] : (g == 1 ? one2 : 0u);
                mma_k16(d, a0, 0u, a2, 0u, b.x, b.y);
                mma_k16(d, a0n, 0u, a2n, 0u, b.z, b.w);
            }
            if (g < 2) {
                // columns 2t, 2t+1 of this lane's row: item ch*IPC (+1 for t >= 2 when IPC == 2)
                int it_c = ch * IPC + ((IPC == 2 && t >= 2) ? 1 : 0);
                if (it_c < items) {
                    const int cc = it_c / GPC, jj = it_c % GPC;
                    const int col0 = IPC == 2 ? 2 * (t & 1) : 2 * t;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (g == 0) {
                            Cx[((size_t)cc * 4 + jj) * 8 + col0 + h] = d[h];
                        } else {
                            const __half vh = __float2half_rn(d[h]);
                            const __half vl = __float2half_rn(d[h] - __half2float(vh));
                            SxB[((size_t)cc * 8 + col0 + h) * 4 + jj] =
                                (uint32_t)__half_as_ushort(vh) | ((uint32_t)__half_as_ushort(vl) << 16);
                            if (GPC == 2) SxB[((size_t)cc * 8 + col0 + h) * 4 + jj + 2] = 0u;
                        }
                    }
                }
            }
        }
        // with M <= 4 the main loop's columns 4..7 repeat columns 0..3: their
        // bias slots must hold finite values (zeros)
        if (MP == 4)
            for (int i = tid; i < ncl * 4 * 4; i += kCons * 32) SxB[(size_t)(i >> 4) * 32 + 16 + (i & 15)] = 0u;
    }
    consumers_sync();

    // ---- main loop: one chunk of the warp's 16 rows per stage ------------------
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, accb[4] = {0.f, 0.f, 0.f, 0.f};
    const int r0 = warp * 16 + g;
    const int jb = t & (GPC - 1);  // bias slot t: group t (gs=64), group t&1 for t < 2 (gs=128)
    constexpr uint32_t R8W = 8 * F::kChunkBytes;  // row r0+8 in the weight tile
    constexpr uint32_t R8S = 8 * GPC * 2;         // row r0+8 in the scale / bias tiles
    uint32_t woff[F::kNW];
#pragma unroll
    for (int v = 0; v < F::kNW; ++v) woff[v] = F::word_off(r0, v, t);
    const uint32_t soff = (uint32_t)(L::kW + r0 * GPC * 2);
    const uint32_t boff = (uint32_t)(L::kW + L::kS + (r0 * GPC + jb) * 2);
    uint32_t bq = bs_a + (uint32_t)((((g & (MP - 1)) * 4) + t) * 16);
    uint32_t cq = cx_a + (uint32_t)(8 * t);
    uint32_t sq = sx_a + (uint32_t)((g * 4 + t) * 4);
    const uint32_t ring_a = smem_addr(ring);
    uint32_t st_a = ring_a;
    int s = 0;
    uint32_t par = 0;
    for (int it = 0; it < ncl; ++it) {
        if (!wait_bounded(smem_addr(&full_bar[s]), par)) break;
        uint32_t w0[F::kNW], w1[F::kNW];
#pragma unroll
        for (int v = 0; v < F::kNW; ++v) {
            w0[v] = lds32(st_a + woff[v]);
            w1[v] = lds32(st_a + woff[v] + R8W);
        }
        // scales of rows r0, r0+8 for the chunk's groups
        uint32_t sw0[GPC / 2], sw1[GPC / 2];
        if constexpr (GPC == 4) {
            const uint2 a = lds64(st_a + soff), b = lds64(st_a + soff + R8S);
            sw0[0] = a.x; sw0[GPC / 2 - 1] = a.y;
            sw1[0] = b.x; sw1[GPC / 2 - 1] = b.y;
        } else {
            sw0[0] = lds32(st_a + soff);
            sw1[0] = lds32(st_a + soff + R8S);
        }
        uint16_t b0, b1;
        if constexpr (HAS_BIAS) {
            b0 = lds16(st_a + boff);
            b1 = lds16(st_a + boff + R8S);
        } else {
            const uint32_t x0 = (jb >> 1) ? sw0[GPC / 2 - 1] : sw0[0];
            const uint32_t x1 = (jb >> 1) ? sw1[GPC / 2 - 1] : sw1[0];
            b0 = __half_as_ushort(sym_bias(__ushort_as_half((uint16_t)(x0 >> (16 * (jb & 1)))), p.ratio));
            b1 = __half_as_ushort(sym_bias(__ushort_as_half((uint16_t)(x1 >> (16 * (jb & 1)))), p.ratio));
        }
        if (GPC == 2 && t >= 2) b0 = b1 = 0;
        // every read of the stage is issued above; release it once the values
        // have arrived (the arrive orders after them)
#pragma unroll
        for (int j = 0; j < GPC; ++j) {
            uint32_t A0[NPR], A1[NPR];
            F::unpack_group(w0, j, t, mg, A0);
            F::unpack_group(w1, j, t, mg, A1);
            float ag[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < MPG; i += 2) {
                const int mi = j * MPG + i;
                const uint4 b = lds128(bq + (uint32_t)((mi >> 1) * MP * 4 * 16));
                mma_k16(ag, A0[2 * i], A1[2 * i], A0[2 * i + 1], A1[2 * i + 1], b.x, b.y);
                mma_k16(ag, A0[2 * i + 2], A1[2 * i + 2], A0[2 * i + 3], A1[2 * i + 3], b.z, b.w);
            }
            const uint2 cxv = lds64(cq + (uint32_t)(j * 32));
            const float cx0 = __uint_as_float(cxv.x), cx1 = __uint_as_float(cxv.y);
            const float sa = (j & 1) ? h2f_hi(sw0[j >> 1]) : h2f_lo(sw0[j >> 1]);
            const float sb = (j & 1) ? h2f_hi(sw1[j >> 1]) : h2f_lo(sw1[j >> 1]);
            acc[0] = fmaf(sa, ag[0] - cx0, acc[0]);
            acc[1] = fmaf(sa, ag[1] - cx1, acc[1]);
            acc[2] = fmaf(sb, ag[2] - cx0, acc[2]);
            acc[3] = fmaf(sb, ag[3] - cx1, acc[3]);
        }
        mma_k8(accb, dup_half(b0), dup_half(b1), lds32(sq));
        mbar_arrive(smem_addr(&empty_bar[s]));
        bq += 8 * MP * 4 * 16;
        cq += 128;
        sq += 128;
        st_a += STAGE;
        if (++s == NST) {
            s = 0;
            par ^= 1u;
            st_a = ring_a;
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] += accb[q];
    const int r1 = r0 + 8;

    // ---- results -------------------------------------------------------------------
    if (S == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = n0 + (q < 2 ? r0 : r1), m = 2 * t + (q & 1);
            if (n < p.N && m < p.M) p.out[(size_t)m * p.N + n] = __float2half_rn(acc[q]);
        }
        return;
    }
    // ranks 1..S-1 store their partials into rank 0's reduction area (not
    // aliased with anything rank 0 may still be using), then one cluster
    // barrier; rank 0 adds them in rank order
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (rank != 0) {
        float *dst = red + (size_t)(rank - 1) * kRowsT * 8;
        st_cluster_v2(smem_addr(dst + r0 * 8 + 2 * t), 0, acc[0], acc[1]);
        st_cluster_v2(smem_addr(dst + r1 * 8 + 2 * t), 0, acc[2], acc[3]);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (rank == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int rr = q < 2 ? r0 : r1, m = 2 * t + (q & 1);
            float v = acc[q];
            for (int k = 1; k < S; ++k) v += red[((size_t)(k - 1) * kRowsT + rr) * 8 + m];
            const int n = n0 + rr;
            if (n < p.N && m < p.M) p.out[(size_t)m * p.N + n] = __float2half_rn(v);
        }
    }
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
    int S, Cs, stages, R;
    uint32_t ring;
    size_t smem;
};

size_t tma_smem(int MP, int Cs, int S, uint32_t ring)
{
    return 1024 + ring + (size_t)Cs * (8 * MP * 4 * 16 + 32 * 4 + 32 * 4) + (size_t)(S - 1) * kRowsT * 8 * 4;
}

template <int FMT, int GS, bool HAS_BIAS, int MP>
int cluster_slots_t(int S, size_t smem)
{
    struct Entry { int dev, S; size_t smem; int slots; };
    static Entry cache[64];
    static int n = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].dev == dev && cache[i].S == S && cache[i].smem == smem) return cache[i].slots;
    auto kern = qmv_tma_kernel<FMT, GS, HAS_BIAS, MP>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudgetT);
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
    if (n < 64) cache[n++] = Entry{dev, S, smem, slots};
    return slots;
}

template <int FMT, int GS, bool HAS_BIAS, int MP>
bool plan_t(int N, int chunks, TPlan &best)
{
    const int R = (N + kRowsT - 1) / kRowsT;
    const int sms = sm_count();
    const uint32_t stage = (uint32_t)Layout<FMT, GS>::stage(HAS_BIAS);
    double best_cost = 1e30;
    bool found = false;
    for (int S = 1; S <= kMaxSplitT && S <= chunks; ++S) {
        const int Cs = (chunks + S - 1) / S;
        if ((S - 1) * Cs >= chunks) continue;
        // ring: as many stages as fit (at most Cs, at most kMaxStagesT)
        const size_t fixed = tma_smem(MP, Cs, S, 0);
        if (fixed + 2 * stage > kSmemBudgetT) continue;
        int st = (int)((kSmemBudgetT - fixed) / stage);
        st = st > kMaxStagesT ? kMaxStagesT : st;
        st = st > Cs ? Cs : st;
        if (st < 1) continue;
        const uint32_t ring = (uint32_t)st * stage;
        const size_t sm = tma_smem(MP, Cs, S, ring);
        if (sm > kSmemBudgetT) continue;
        const int slots = S == 1 ? 2 * sms : cluster_slots_t<FMT, GS, HAS_BIAS, MP>(S, sm);
        if (slots <= 0) continue;
        const int waves = (R + slots - 1) / slots;
        // time ~ waves x (chunks per CTA + prologue/epilogue worth ~3 chunks)
        const double cost = (double)waves * (Cs + 3) + 0.05 * S;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = TPlan{S, Cs, st, R, ring, sm};
            found = true;
        }
    }
    return found;
}

template <int FMT, int GS, bool HAS_BIAS, int MP>
int launch_t(const TmaParams &p0, const CUtensorMap &map, int chunks, cudaStream_t s)
{
    TPlan pl;
    if (!plan_t<FMT, GS, HAS_BIAS, MP>(p0.N, chunks, pl)) return BQD_ERR_UNSUPPORTED;
    TmaParams p = p0;
    p.S = pl.S;
    p.Cs = pl.Cs;
    p.stages = pl.stages;
    p.ring_bytes = pl.ring;
    if (getenv("BQD_DEBUG_PLAN"))
        fprintf(stderr, "bqd tma plan: N=%d K=%d M=%d gs=%d -> S=%d Cs=%d stages=%d R=%d grid=%d smem=%zu\n", p.N, p.K,
                p.M, GS, pl.S, pl.Cs, pl.stages, pl.R, pl.R * pl.S, pl.smem);
    auto kern = qmv_tma_kernel<FMT, GS, HAS_BIAS, MP>;
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudgetT) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.R * pl.S);
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
    return cudaLaunchKernelEx(&cfg, kern, map, p) == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
}

template <int FMT, int GS>
int launch_fmt_gs(const TmaParams &p, const CUtensorMap &map, int chunks, bool has_bias, int MP, cudaStream_t s)
{
    if (MP == 4)
        return has_bias ? launch_t<FMT, GS, true, 4>(p, map, chunks, s) : launch_t<FMT, GS, false, 4>(p, map, chunks, s);
    return has_bias ? launch_t<FMT, GS, true, 8>(p, map, chunks, s) : launch_t<FMT, GS, false, 8>(p, map, chunks, s);
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
    // whole 256-code chunks; TMA needs 16-byte aligned rows and base; cp.async
    // of a chunk's scales needs 4/8-byte alignment
    if (a.K % kChunkT != 0 || a.row_bytes % 16 != 0) return BQD_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(a.w) & 15) || (reinterpret_cast<uintptr_t>(a.x) & 15)) return BQD_ERR_UNSUPPORTED;
    const uintptr_t salign = (uintptr_t)(kChunkT / a.gs) * 2;
    if ((reinterpret_cast<uintptr_t>(a.scales) & (salign - 1)) ||
        (a.biases && (reinterpret_cast<uintptr_t>(a.biases) & (salign - 1))))
        return BQD_ERR_UNSUPPORTED;
    if (a.K > (int64_t)1 << 28 || a.N > (int64_t)1 << 28) return BQD_ERR_UNSUPPORTED;
    auto enc = encode_fn();
    if (!enc) return BQD_ERR_UNSUPPORTED;

    const bool b64 = a.fmt == BQD_FMT_AFFINE2;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)a.row_bytes, (cuuint64_t)a.N};
    cuuint64_t strides[1] = {(cuuint64_t)a.row_bytes};
    cuuint32_t box[2] = {b64 ? 64u : 32u, (cuuint32_t)kRowsT};
    cuuint32_t estr[2] = {1, 1};
    CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.w), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, b64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return BQD_ERR_CUDA;

    TmaParams p;
    p.scales = a.scales; p.biases = a.biases; p.ratio = a.ratio;
    p.N = (int)a.N; p.K = (int)a.K; p.G = (int)a.G;
    p.chunks = (int)(a.K / kChunkT);
    p.zero = 0;
    p.S = p.Cs = p.stages = 0;
    p.ring_bytes = 0;
    const bool hb = a.biases != nullptr;
    for (int64_t m0 = 0; m0 < a.M; m0 += 8) {
        const int M = (int)((a.M - m0) < 8 ? (a.M - m0) : 8);
        const int MP = M <= 4 ? 4 : 8;
        p.M = M;
        p.x = a.x + m0 * a.K;
        p.out = a.out + m0 * a.N;
        int st;
        if (b64)
            st = a.gs == 64 ? launch_fmt_gs<BQD_FMT_AFFINE2, 64>(p, map, p.chunks, hb, MP, s)
                            : launch_fmt_gs<BQD_FMT_AFFINE2, 128>(p, map, p.chunks, hb, MP, s);
        else
            st = a.gs == 64 ? launch_fmt_gs<BQD_FMT_AFFINE1, 64>(p, map, p.chunks, hb, MP, s)
                            : launch_fmt_gs<BQD_FMT_AFFINE1, 128>(p, map, p.chunks, hb, MP, s);
        if (st != BQD_OK) return st;
    }
    return BQD_OK;
}

}  // namespace bqd
