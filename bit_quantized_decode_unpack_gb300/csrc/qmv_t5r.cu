// Tensor-core decode QMV for t5 ternary weights fed by TMA into a shared-memory
// ring (M <= 5 activation rows per pass, K a multiple of 1024).
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" -- §二.3 (t5:
// trits {0,1,2}, five per uint8, 13 bytes per 64-weight group / 26 per
// 128-weight group), §二.2 (one read of every weight byte serves all M rows;
// the sym variant rebuilds the bias from the scale).
//
// Arithmetic as in the register-streaming t5 kernel: a 256-entry shared table
// maps a byte to its five trits as 2-bit fields (bits 0,2,4,6,8); byte i of
// group 2b is paired with byte i of group 2b+1 (gs=64) or byte i with byte
// i+26 (gs=128); per trit one LOP3 (mask + magic exponent) and one HFMA2
// give fp16(s*t) for both halves; mma.sync m16n8k16 with fp32 accumulation
// (weight rows = MMA rows, x rows = MMA columns); the bias term is an extra
// MMA against the group sums of x split into fp16 high part and remainder.
// A thread's slice of a row chunk is 52 bytes (4 groups of 64 / 2 of 128),
// i.e. codes [256t, 256t+256) of the chunk.
//
// CTA: 8 consumer warps (warp w owns weight rows n0+16w .. +15) and one
// producer warp.  Per ring stage (one 1024-code chunk of the CTA's 128 rows)
// the producer issues three 2-D TMA copies -- weights [128][208 B], scales
// and biases [128][groups of the chunk] -- and, from the chunk of x (TMA into
// a double buffer, one chunk ahead), builds the MMA B fragments and the
// group sums.  Weights,
// scales and biases are requested before the programmatic-dependent-launch
// wait.  K is split over the S CTAs of a cluster; the partial sums are
// reduce-scattered through distributed shared memory, each rank adding its
// slice of rows in rank order (deterministic, no global scratch).  Every
// mbarrier wait is bounded; an expiry is counted for bqd_device_status.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "bqd_internal.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

__device__ unsigned int g_qmv_t5r_timeouts = 0;

constexpr int kConsR = 8;                      // consumer warps
constexpr int kThreadsR = (kConsR + 1) * 32;   // + one producer warp
constexpr int kRowsR = 16 * kConsR;            // weight rows per CTA
constexpr int kCodesR = 1024;                  // codes per row per stage
constexpr int kBytesR = 208;                   // t5 bytes per row per stage
constexpr int kMmasR = 65;                     // per 16-row unit: 26 byte pairs x 5 trits x 2 / 8
constexpr int kPairsR = 33;                    // MMA pairs (the last one half empty)
constexpr int kMaxMR = 5;                      // x rows per pass
constexpr int kMaxStagesR = 4;
constexpr int kMaxSplitR = 16;
constexpr size_t kSmemBudgetR = 108 * 1024;    // two CTAs per SM, with the static tables and the 1 KB reserve

struct T5RParams {
    const __half *x;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M;     // x rows per pass (the staging and fragment layouts)
    int Mtot;  // x rows of the call; pass blockIdx.y takes rows M*y .. M*y+M-1
    int N, K, G, chunks, S, Cs, stages, RS;
    uint32_t stage_bytes;
    uint32_t zero;  // always 0: keeps the magic constants opaque (in registers)
    unsigned long long wait_ns;  // limit of the pipeline waits
};

template <int GS>
struct G5 {
    static constexpr int B = GS == 64 ? 13 : 26;     // bytes per group
    static constexpr int NG = GS == 64 ? 4 : 2;      // groups per thread slice
    static constexpr int NB = GS == 64 ? 2 : 1;      // bias MMAs per chunk
    static constexpr int GPC = kCodesR / GS;         // groups per chunk
    // pair j (0..25) of a slice: byte a (group 2*beta) with byte a + B (group 2*beta+1)
    __host__ __device__ static constexpr int beta(int j) { return j / B; }
    __host__ __device__ static constexpr int byte_a(int j) { return 2 * B * (j / B) + j % B; }
    // code of the chunk behind half `hi` of half2 h of slot t's slice, or -1 (padding trit)
    __host__ __device__ static constexpr int code(int h, int hi, int t)
    {
        const int j = h / 5, d = h % 5;
        const int o = byte_a(j) + hi * B;
        const int grp = o / B, bg = o % B;
        const int within = 5 * bg + d;
        return within < GS ? (NG * t + grp) * GS + within : -1;
    }
};

// stage layout: weights [128][208] | scales [128][GPC] | biases (if any) | B fragments [33][M][4] uint4
// | group sums [NB][M][4] uint2
template <int GS, bool HAS_BIAS>
struct Stage5 {
    static constexpr int kW = kRowsR * kBytesR;
    static constexpr int kS = kRowsR * G5<GS>::GPC * 2;
    static constexpr int kScale = kW;
    static constexpr int kBias = kW + kS;
    static constexpr int kB = kW + kS * (HAS_BIAS ? 2 : 1);
    __host__ __device__ static constexpr int sx_off(int M) { return kB + kPairsR * M * 64; }
    __host__ __device__ static constexpr int bytes(int M) { return (sx_off(M) + G5<GS>::NB * M * 32 + 127) / 128 * 128; }
};

// pipeline waits give up after the call's limit; drain waits after a second
__device__ __forceinline__ bool wait_bounded_r(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    return mbar_wait_for(bar, parity, limit_ns, &g_qmv_t5r_timeouts);
}

__device__ __forceinline__ void mbar_arrive_r(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint4 lds128r(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ void mma_r(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void st_cluster_v2r(uint32_t local_addr, uint32_t rank, float a, float b)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(a), "f"(b) : "memory");
}

template <int GS, bool HAS_BIAS>
__global__ void __launch_bounds__(kThreadsR, 2)
    qmv_t5r_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap bmap, const __grid_constant__ CUtensorMap xmap, const T5RParams p)
{
    using Ge = G5<GS>;
    using SL = Stage5<GS, HAS_BIAS>;
    constexpr int B = Ge::B;
    constexpr int GPC = Ge::GPC;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStagesR], empty_bar[kMaxStagesR], x_bar[2];
    __shared__ uint32_t lut[256];
    __shared__ __align__(16) uint16_t koff[kPairsR * 4 * 8];  // (pair, slot) -> staging offsets of its 8 codes

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int S = p.S;
    const int rank = S > 1 ? (int)cluster_ctarank() : 0;
    const int n0 = (blockIdx.x / S) * kRowsR;
    const int c_lo = rank * p.Cs;
    const int ncl = max(0, min(p.Cs, p.chunks - c_lo));
    const int NST = p.stages;
    const int M = p.M;
    const uint32_t STB = p.stage_bytes;

    // the next kernel may launch now: it only prefetches its weights until
    // its griddepcontrol.wait, which waits for this whole grid
    pdl_launch_dependents();
    if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_a = smem_addr(smem);
    const uint32_t xraw_a = ring_a + (uint32_t)NST * STB;  // 2 x [M][1024] fp16, producer only
    const uint32_t XB = (uint32_t)(M * kCodesR * 2);
    float *red = reinterpret_cast<float *>(smem + (size_t)NST * STB + 2 * (size_t)XB);  // [S][RS][8]

    // decode table: byte -> five trits at bits 0,2,4,6,8 (invalid bytes -> 0)
    if (tid < 256) {
        int v = tid, e = 0;
        if (v < 243) {
#pragma unroll
            for (int d = 0; d < 5; ++d) {
                e |= (v % 3) << (2 * d);
                v /= 3;
            }
        }
        lut[tid] = (uint32_t)e;
    }
    for (int e = tid; e < kPairsR * 4 * 8; e += kThreadsR) {
        const int q = e & 7, slot = (e >> 3) & 3, ip = e >> 5;
        const int i = 2 * ip + (q >> 2);  // MMA index
        const int qq = q & 3, sl = qq >> 1, hi = qq & 1;
        // staging layout [box k/256][row m][256] fp16: code k of row m sits at
        // this offset + 512 m.  Padding trits point at code 0: their A entries
        // are constant zeros, so only a finite x value is needed there.
        const int kc = i < kMmasR ? Ge::code(2 * i + sl, hi, slot) : -1;
        koff[e] = (uint16_t)(kc < 0 ? 0 : ((kc >> 8) * M * 512 + (kc & 255) * 2));
    }
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 33);  // producer lane 0 (expect_tx) + 32 once x is prepared
            mbar_init(smem_addr(&empty_bar[s]), kConsR * 32);
        }
        mbar_init(smem_addr(&x_bar[0]), 1);
        mbar_init(smem_addr(&x_bar[1]), 1);
    }
    __syncthreads();

    if (warp == kConsR) {
        // ---- producer ----------------------------------------------------------------
        auto issue = [&](int it, int s) {
            if (lane == 0) {
                const uint32_t bar = smem_addr(&full_bar[s]);
                const uint32_t st = ring_a + (uint32_t)s * STB;
                mbar_arrive_expect_tx(bar, (uint32_t)(SL::kW + SL::kS * (HAS_BIAS ? 2 : 1)));
                const int c = c_lo + it;
                tma_2d(st, &wmap, c * kBytesR, n0, bar);
                tma_2d(st + SL::kScale, &smap, c * GPC, n0, bar);
                if (HAS_BIAS) tma_2d(st + SL::kBias, &bmap, c * GPC, n0, bar);
            }
        };
        // x of chunk `it` (four 256-code boxes of M rows) into staging buffer it & 1
        auto issue_x = [&](int it) {
            if (lane == 0) {
                const uint32_t bar = smem_addr(&x_bar[it & 1]);
                mbar_arrive_expect_tx(bar, XB);
                const int k0 = (c_lo + it) * kCodesR;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tma_2d(xraw_a + (uint32_t)(it & 1) * XB + (uint32_t)(j * 512 * M), &xmap, k0 + 256 * j,
                           M * (int)blockIdx.y, bar);
            }
        };
        const int pre = min(NST, ncl);
        for (int it = 0; it < pre; ++it) issue(it, it);
        pdl_wait();
        if (ncl > 0) issue_x(0);
        int s = 0, done = 0, issued_w = pre;
        uint32_t par = 0;
        for (int it = 0; it < ncl; ++it) {
            const uint32_t st = ring_a + (uint32_t)s * STB;
            if (it >= NST) {
                bool ok = lane == 0 ? wait_bounded_r(smem_addr(&empty_bar[s]), par ^ 1u, p.wait_ns) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                issue(it, s);
                issued_w = it + 1;
            }
            {
                bool ok = lane == 0 ? wait_bounded_r(smem_addr(&x_bar[it & 1]), (it >> 1) & 1, p.wait_ns) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            // the other buffer was last read while preparing chunk it-1 (finished,
            // see the __syncwarp below): order those reads before the next copy
            fence_proxy_async_smem();
            if (it + 1 < ncl) issue_x(it + 1);
            // staging buffer: box j holds rows 0..M-1 of codes [256 j, 256 j + 256)
            const uint32_t xb = xraw_a + (uint32_t)(it & 1) * XB;
            // B fragments: entry (pair ip, column m, slot) = two MMAs' (b0, b1)
            for (int e = lane; e < kPairsR * 4; e += 32) {
                const int ip = e >> 2, slot = e & 3;
                const uint4 kw = lds128r(smem_addr(&koff[e * 8]));
                const uint32_t o[8] = {xb + (kw.x & 0xffffu), xb + (kw.x >> 16), xb + (kw.y & 0xffffu), xb + (kw.y >> 16),
                                       xb + (kw.z & 0xffffu), xb + (kw.z >> 16), xb + (kw.w & 0xffffu), xb + (kw.w >> 16)};
                const uint32_t dst = st + SL::kB + (uint32_t)((ip * M * 4 + slot) * 16);
#pragma unroll
                for (int m = 0; m < kMaxMR; ++m) {
                    if (m < M) {
                        uint32_t h[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            uint16_t v16;
                            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v16) : "r"(o[q] + (uint32_t)(512 * m)));
                            h[q] = v16;
                        }
                        sts128(dst + (uint32_t)(64 * m), make_uint4(__byte_perm(h[0], h[1], 0x5410), __byte_perm(h[2], h[3], 0x5410),
                                                                   __byte_perm(h[4], h[5], 0x5410), __byte_perm(h[6], h[7], 0x5410)));
                    }
                }
            }
            __syncwarp();
            // group sums on the tensor core: A row r is the indicator of group r
            // (zero at padding trits), B the fragments just built, so D[r][m] =
            // Sx[r][m]; lane (g, t) holds groups g, g+8 x columns 2t, 2t+1
            {
                uint32_t P[2][2];
#pragma unroll
                for (int be = 0; be < 2; ++be)
#pragma unroll
                    for (int rh = 0; rh < 2; ++rh) {
                        const int row = g + 8 * rh, ga = Ge::NG * t + 2 * be;
                        P[be][rh] = (ga == row ? 0x3C00u : 0u) | (ga + 1 == row ? 0x3C000000u : 0u);
                    }
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t bq = st + SL::kB + (uint32_t)((min(g, M - 1) * 4 + t) * 16);
                uint4 bv = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int i = 0; i < kMmasR; ++i) {
                    if ((i & 1) == 0) bv = lds128r(bq + (uint32_t)((i >> 1) * M * 64));
                    const int h0 = 2 * i, h1 = 2 * i + 1;
                    const bool pad0 = 5 * ((h0 / 5) % B) + h0 % 5 >= GS, pad1 = 5 * ((h1 / 5) % B) + h1 % 5 >= GS;
                    const int be0 = Ge::beta(h0 / 5), be1 = Ge::beta(h1 / 5);
                    const uint32_t a0 = pad0 ? 0u : P[be0][0], a1 = pad0 ? 0u : P[be0][1];
                    const uint32_t a2 = pad1 ? 0u : P[be1][0], a3 = pad1 ? 0u : P[be1][1];
                    mma_r((i & 1) ? d1 : d0, a0, a1, a2, a3, (i & 1) ? bv.z : bv.x, (i & 1) ? bv.w : bv.y);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = g + 8 * (q >> 1), m = 2 * t + (q & 1);
                    if (r < GPC && m < M) {
                        const float v = d0[q] + d1[q];
                        const __half hi = __float2half_rn(v);
                        const __half lo = __float2half_rn(v - __half2float(hi));
                        const int slot = r / Ge::NG, rem = r % Ge::NG, nb = rem >> 1, s_ = rem & 1;
                        const uint32_t a = st + (uint32_t)SL::sx_off(M) + (uint32_t)(((nb * M + m) * 4 + slot) * 8 + 4 * s_);
                        asm volatile("st.shared.u32 [%0], %1;" ::"r"(a),
                                     "r"((uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16))
                                     : "memory");
                    }
                }
            }
            __syncwarp();  // the staging area is rewritten by the next chunk
            mbar_arrive_r(smem_addr(&full_bar[s]));
            done = it + 1;
            if (++s == NST) {
                s = 0;
                par ^= 1u;
            }
        }
        // every copy this CTA issued has landed before anyone leaves: stages whose
        // weights were requested but that were never prepared (a wait expired)
        // get their missing arrivals, then the last stages are awaited; the x
        // copy of chunk `done` is in flight whenever the loop stopped early
        for (int it = done; it < issued_w; ++it) mbar_arrive_r(smem_addr(&full_bar[it % NST]));
        if (lane == 0) {
            for (int it = max(0, issued_w - NST); it < issued_w; ++it)
                wait_bounded_r(smem_addr(&full_bar[it % NST]), (it / NST) & 1, kDrainWaitNs);
            if (done < ncl) wait_bounded_r(smem_addr(&x_bar[done & 1]), (done >> 1) & 1, kDrainWaitNs);
        }
        __syncwarp();
        if (S > 1) {
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        }
        return;
    }

    // ---- consumers -------------------------------------------------------------------
    uint32_t mg[5];
#pragma unroll
    for (int d = 0; d < 5; ++d) mg[d] = magic(2 * d) ^ p.zero;
    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
    const int mcol = min(g, M - 1);  // columns >= M read a valid column; their outputs are dropped
    const int r0 = warp * 16 + g;
    uint32_t st_a = ring_a;
    int s = 0;
    uint32_t par = 0;
    for (int it = 0; it < ncl; ++it) {
        if (!wait_bounded_r(smem_addr(&full_bar[s]), par, p.wait_ns)) break;
        // this lane's 52-byte slices of rows r0 and r0+8
        uint32_t wa[13], wb[13];
#pragma unroll
        for (int q = 0; q < 13; ++q) {
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wa[q]) : "r"(st_a + (uint32_t)(r0 * kBytesR + 52 * t + 4 * q)));
            asm volatile("ld.shared.u32 %0, [%1];"
                         : "=r"(wb[q])
                         : "r"(st_a + (uint32_t)((r0 + 8) * kBytesR + 52 * t + 4 * q)));
        }
        // scales (and biases) of this slice's groups, rows r0 and r0+8
        uint16_t sv[2][Ge::NG], bv[2][Ge::NG];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t sa = st_a + SL::kScale + (uint32_t)(((r0 + 8 * rr) * GPC + Ge::NG * t) * 2);
            uint32_t sw[2] = {0u, 0u}, bw[2] = {0u, 0u};
            if (Ge::NG == 4) {
                asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(sw[0]), "=r"(sw[1]) : "r"(sa));
                if (HAS_BIAS)
                    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(bw[0]), "=r"(bw[1]) : "r"(sa + SL::kS));
            } else {
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sw[0]) : "r"(sa));
                if (HAS_BIAS) asm volatile("ld.shared.u32 %0, [%1];" : "=r"(bw[0]) : "r"(sa + SL::kS));
            }
#pragma unroll
            for (int q = 0; q < Ge::NG; ++q) {
                sv[rr][q] = (uint16_t)(sw[q >> 1] >> (16 * (q & 1)));
                bv[rr][q] = HAS_BIAS ? (uint16_t)(bw[q >> 1] >> (16 * (q & 1)))
                                     : __half_as_ushort(sym_bias(__ushort_as_half(sv[rr][q]), p.ratio));
            }
        }
        // per pair-block beta: s2 = (s[2b], s[2b+1]) and c_d = -2^(10-2d) * s2
        constexpr int NBETA = GS == 64 ? 2 : 1;
        uint32_t s2[2][NBETA], cst[2][NBETA][5];
        bool fast = true;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int be = 0; be < NBETA; ++be) {
                s2[rr][be] = (uint32_t)sv[rr][2 * be] | ((uint32_t)sv[rr][2 * be + 1] << 16);
#pragma unroll
                for (int d = 0; d < 5; ++d)
                    cst[rr][be][d] =
                        hmul2(s2[rr][be], dup_half(__half_as_ushort(__float2half_rn(-(float)(1024 >> (2 * d))))));
                // the constants stay finite for |s| < 63; else the exact (magic - offset) * s form
                fast = fast && fabsf(__half2float(__ushort_as_half(sv[rr][2 * be]))) < 63.f &&
                       fabsf(__half2float(__ushort_as_half(sv[rr][2 * be + 1]))) < 63.f;
            }
        const bool all_fast = __all_sync(0xffffffffu, fast);
        const uint32_t bq = st_a + SL::kB + (uint32_t)((mcol * 4 + t) * 16);
        const uint32_t bstride = (uint32_t)(M * 64);

        auto pairs = [&](auto fast_tag) {
            constexpr bool kFast = decltype(fast_tag)::value;
            uint4 bcur = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int jp = 0; jp < 13; ++jp) {
                uint32_t A0[10], A1[10];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * jp + jj;
                    const int oa = Ge::byte_a(j), ob = oa + B;
                    const int be = Ge::beta(j);
                    const uint32_t la0 = lut[__byte_perm(wa[oa >> 2], 0, 0x4440 | (oa & 3))];
                    const uint32_t lb0 = lut[__byte_perm(wa[ob >> 2], 0, 0x4440 | (ob & 3))];
                    const uint32_t la1 = lut[__byte_perm(wb[oa >> 2], 0, 0x4440 | (oa & 3))];
                    const uint32_t lb1 = lut[__byte_perm(wb[ob >> 2], 0, 0x4440 | (ob & 3))];
                    const uint32_t v0 = mad_u32(lb0, 65536u, la0);
                    const uint32_t v1 = mad_u32(lb1, 65536u, la1);
#pragma unroll
                    for (int d = 0; d < 5; ++d) {
                        if (5 * (j % B) + d >= GS) {  // padding trit of a group's last byte
                            A0[5 * jj + d] = A1[5 * jj + d] = 0u;
                            continue;
                        }
                        const uint32_t mask = 0x00030003u << (2 * d);
                        const uint32_t h0 = (v0 & mask) | mg[d];
                        const uint32_t h1 = (v1 & mask) | mg[d];
                        if (kFast) {
                            A0[5 * jj + d] = hfma2(h0, s2[0][be], cst[0][be][d]);
                            A1[5 * jj + d] = hfma2(h1, s2[1][be], cst[1][be][d]);
                        } else {
                            A0[5 * jj + d] = hmul2(hsub2(h0, mg[d]), s2[0][be]);
                            A1[5 * jj + d] = hmul2(hsub2(h1, mg[d]), s2[1][be]);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 5; ++q) {
                    const int i = 5 * jp + q;
                    if ((i & 1) == 0) bcur = lds128r(bq + (uint32_t)(i >> 1) * bstride);
                    const uint32_t b0 = (i & 1) ? bcur.z : bcur.x, b1 = (i & 1) ? bcur.w : bcur.y;
                    mma_r(acc[i & 3], A0[2 * q], A1[2 * q], A0[2 * q + 1], A1[2 * q + 1], b0, b1);
                }
            }
        };
        if (all_fast) pairs(std::true_type{});
        else pairs(std::false_type{});
        // bias term: slots 2t, 2t+1 <- group NG t + 2nb, slots 2t+8, 2t+9 <- group NG t + 2nb + 1
        const uint32_t sq = st_a + (uint32_t)SL::sx_off(M) + (uint32_t)((mcol * 4 + t) * 8);
#pragma unroll
        for (int nb = 0; nb < Ge::NB; ++nb) {
            uint32_t bx, by;
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(bx), "=r"(by) : "r"(sq + (uint32_t)(nb * M * 32)));
            mma_r(acc[nb & 3], dup_half(bv[0][2 * nb]), dup_half(bv[1][2 * nb]), dup_half(bv[0][2 * nb + 1]),
                  dup_half(bv[1][2 * nb + 1]), bx, by);
        }
        mbar_arrive_r(smem_addr(&empty_bar[s]));
        st_a += STB;
        if (++s == NST) {
            s = 0;
            par ^= 1u;
            st_a = ring_a;
        }
    }
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = (acc[0][q] + acc[1][q]) + (acc[2][q] + acc[3][q]);

    // ---- results: value q is row r0 + 8 (q >> 1), column 2t + (q & 1) -------------------
    const int Mv = min(M, p.Mtot - M * (int)blockIdx.y);  // rows of this pass that exist
    __half *outg = p.out + (size_t)(M * blockIdx.y) * p.N;
    if (S == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = n0 + r0 + 8 * (q >> 1), m = 2 * t + (q & 1);
            if (n < p.N && m < Mv) outg[(size_t)m * p.N + n] = __float2half_rn(v[q]);
        }
        return;
    }
    const int RS = p.RS;
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = r0 + 8 * h;
        const int q = row / RS;
        st_cluster_v2r(smem_addr(red + ((size_t)rank * RS + (row - q * RS)) * 8 + 2 * t), (uint32_t)q, v[2 * h],
                       v[2 * h + 1]);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    const int row0 = rank * RS;
    const int nrow = min(RS, kRowsR - row0);
    for (int e = tid; e < nrow * M; e += kConsR * 32) {
        const int lr = e / M, m = e % M;
        float sum = 0.f;
        for (int k = 0; k < S; ++k) sum += red[((size_t)k * RS + lr) * 8 + m];
        const int n = n0 + row0 + lr;
        if (n < p.N && m < Mv) outg[(size_t)m * p.N + n] = __float2half_rn(sum);
    }
}

// ---- host side -----------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_r()
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

bool encode_2d(CUtensorMap &map, CUtensorMapDataType dt, const void *base, int64_t cols, int64_t rows,
               int64_t row_bytes, int box_cols, int box_rows = kRowsR)
{
    auto enc = encode_fn_r();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(&map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

struct RPlan {
    int S, Cs, stages, R, RS;
    size_t smem;
};

template <int GS, bool HAS_BIAS>
size_t t5r_smem(int M, int S, int stages, int RS)
{
    return 1024 + (size_t)stages * Stage5<GS, HAS_BIAS>::bytes(M) + 2 * (size_t)M * kCodesR * 2 + (size_t)S * RS * 8 * 4;
}

template <int GS, bool HAS_BIAS>
int cluster_slots_r(int S, size_t smem)
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
    auto kern = qmv_t5r_kernel<GS, HAS_BIAS>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudgetR);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(kThreadsR);
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
template <int GS, bool HAS_BIAS>
bool plan_r(int M, int N, int chunks, int P, RPlan &best)
{
    const int R = (N + kRowsR - 1) / kRowsR;
    const int sms = sm_count();
    const size_t stage = Stage5<GS, HAS_BIAS>::bytes(M);
    double best_cost = 1e30;
    bool found = false;
    for (int S = 1; S <= kMaxSplitR && S <= chunks; ++S) {
        const int Cs = (chunks + S - 1) / S;
        if ((S - 1) * Cs >= chunks) continue;
        const int RS = (kRowsR + S - 1) / S;
        const size_t fixed = t5r_smem<GS, HAS_BIAS>(M, S, 0, RS);
        if (fixed + stage > kSmemBudgetR) continue;
        int st = (int)((kSmemBudgetR - fixed) / stage);
        st = std::min(st, kMaxStagesR);
        st = std::min(st, Cs);
        if (st < 1) continue;
        const size_t sm = t5r_smem<GS, HAS_BIAS>(M, S, st, RS);
        const int slots = S == 1 ? 2 * sms : cluster_slots_r<GS, HAS_BIAS>(S, sm);
        if (slots <= 0) continue;
        const int waves = (R * P + slots - 1) / slots;
        // time ~ waves x (chunks per CTA + first-stage latency and reduction,
        // ~1 chunk); a single-stage ring (no overlap of copy and compute) costs
        // about twice as much per chunk
        const double per_chunk = (st < 2 && Cs > 1) ? 2.0 : 1.0;
        const double cost = (double)waves * (Cs * per_chunk + 1) + 0.05 * S;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = RPlan{S, Cs, st, R, RS, sm};
            found = true;
        }
    }
    return found;
}

template <int GS, bool HAS_BIAS>
int launch_r(const T5RParams &p0, const CUtensorMap &wmap, cudaStream_t s)
{
    RPlan pl;
    const int P = (p0.Mtot + p0.M - 1) / p0.M;
    if (!plan_r<GS, HAS_BIAS>(p0.M, p0.N, p0.chunks, P, pl)) return BQD_ERR_UNSUPPORTED;
    T5RParams p = p0;
    p.S = pl.S;
    p.Cs = pl.Cs;
    p.stages = pl.stages;
    p.RS = pl.RS;
    p.stage_bytes = (uint32_t)Stage5<GS, HAS_BIAS>::bytes(p.M);
    constexpr int GPC = G5<GS>::GPC;
    CUtensorMap smap, bmap;
    if (!encode_2d(smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.scales, p.G, p.N, (int64_t)p.G * 2, GPC)) return BQD_ERR_CUDA;
    bmap = smap;
    if (HAS_BIAS && !encode_2d(bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.biases, p.G, p.N, (int64_t)p.G * 2, GPC))
        return BQD_ERR_CUDA;
    // x: [Mtot][K] fp16, box {256 codes, M rows}; a pass's rows past Mtot read as zeros
    CUtensorMap xmap;
    if (!encode_2d(xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.x, p.K, p.Mtot, (int64_t)p.K * 2, 256, p.M))
        return BQD_ERR_CUDA;
    if (opt_debug_plan())
        fprintf(stderr, "bqd t5r plan: N=%d K=%d M=%d (%d per pass) gs=%d -> S=%d Cs=%d stages=%d R=%d grid=%dx%d smem=%zu\n",
                p.N, p.K, p.Mtot, p.M, GS, pl.S, pl.Cs, pl.stages, pl.R, pl.R * pl.S, P, pl.smem);
    auto kern = qmv_t5r_kernel<GS, HAS_BIAS>;
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudgetR) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.R * pl.S, P);
    cfg.blockDim = dim3(kThreadsR);
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
    return cudaLaunchKernelEx(&cfg, kern, wmap, smap, bmap, xmap, p) == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
}

}  // namespace

int take_qmv_t5r_timeouts(unsigned int *count)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmv_t5r_timeouts, sizeof(v)) != cudaSuccess) return BQD_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_qmv_t5r_timeouts, &zero, sizeof(zero)) != cudaSuccess) return BQD_ERR_CUDA;
    *count = v;
    return BQD_OK;
}

int launch_qmv_t5r(const QmvArgs &a, cudaStream_t s)
{
    if (a.fmt != BQD_FMT_T5) return BQD_ERR_UNSUPPORTED;
    // whole 1024-code chunks (208 bytes per row: 16-byte multiple), 16-byte
    // aligned bases and scale rows (K/gs a multiple of 8 for the TMA boxes)
    if (a.K % kCodesR != 0 || a.row_bytes % 16 != 0 || a.G % 8 != 0) return BQD_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(a.w) & 15) || (reinterpret_cast<uintptr_t>(a.x) & 15) ||
        (reinterpret_cast<uintptr_t>(a.scales) & 15) || (a.biases && (reinterpret_cast<uintptr_t>(a.biases) & 15)))
        return BQD_ERR_UNSUPPORTED;
    if (a.K > (int64_t)1 << 28 || a.N > (int64_t)1 << 28) return BQD_ERR_UNSUPPORTED;
    CUtensorMap wmap;
    if (!encode_2d(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, a.row_bytes, a.N, a.row_bytes, kBytesR))
        return BQD_ERR_UNSUPPORTED;
    T5RParams p;
    p.scales = a.scales; p.biases = a.biases; p.ratio = a.ratio;
    p.N = (int)a.N; p.K = (int)a.K; p.G = (int)a.G;
    p.chunks = (int)(a.K / kCodesR);
    p.zero = 0;
    p.wait_ns = (unsigned long long)opt_wait_ns();
    p.S = p.Cs = p.stages = p.RS = 0;
    p.stage_bytes = 0;
    const bool hb = a.biases != nullptr;
    // passes of at most kMaxMR x rows, all in one launch (grid row y = rows
    // kMaxMR*y ..): the fixed cost of a call is paid once and later passes find
    // the weights in L2
    if (a.M > (int64_t)kMaxMR * 65535) return BQD_ERR_UNSUPPORTED;
    p.M = (int)(a.M < kMaxMR ? a.M : kMaxMR);
    p.Mtot = (int)a.M;
    p.x = a.x;
    p.out = a.out;
    if (a.gs == 64) return hb ? launch_r<64, true>(p, wmap, s) : launch_r<64, false>(p, wmap, s);
    return hb ? launch_r<128, true>(p, wmap, s) : launch_r<128, false>(p, wmap, s);
}

}  // namespace bqd
