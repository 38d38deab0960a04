// Tensor-core decode QMV for t5 ternary weights, M <= 8 rows of x.
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" -- §二.3 (t5:
// trits {0,1,2}, five per uint8, 13 bytes per 64-weight group / 26 per
// 128-weight group; decode with bonsai_t5_qmv / bonsai_t5_qmv_wide), §二.2
// (one read of every weight byte serves all M rows).
//
// Same arithmetic as the 1/2-bit kernel: A = fp16(s*t) on the tensor cores,
// the bias term (sym: -ratio*s, default ratio 1, i.e. w = s*t - s) as a small
// extra MMA on split-precision group sums of x.  What differs is the weight
// geometry: t5 groups are 13 (or 26) bytes, so the unit of work is 16 weight
// rows x 208 bytes (16 groups of 64 or 8 groups of 128, 1024 codes), a
// thread's slice is 52 bytes (4 or 2 whole groups), and slices are not
// 16-byte aligned.  Each warp therefore streams its units into a private
// two-stage shared-memory ring with bulk (TMA) copies, one 208-byte copy per
// row, completion tracked by an mbarrier; lanes then read their slices with
// 32-bit shared loads.
//
// Decode: a 256-entry shared table maps a byte to its five trits as 2-bit
// fields (bits 0,2,4,6,8).  Byte i of group 2b is paired with byte i of group
// 2b+1 (gs=64) or byte i with byte i+26 (gs=128): one table lookup per byte,
// one multiply-add to place the partner's fields in the high half, then per
// trit one LOP3 (mask + magic exponent) and one HFMA2 (s*t with per-half
// scales).  A group's last byte carries padding trits (0), whose B entries
// are 0.
#include <stdio.h>
#include <stdlib.h>

#include <mutex>
#include <type_traits>

#include "bqd_internal.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

constexpr int kThreads = kWarps * 32;
constexpr int kMaxM = 8;
constexpr int kMaxTc = 8;
constexpr int kChunkBytes = 208;  // per weight row and unit
constexpr int kChunkCodes = 1024;
constexpr int kSliceWords = 13;   // 52 bytes per thread
constexpr int kMmas = 65;         // per unit: 26 byte pairs x 5 trits x 2 halves / 8 per MMA row
constexpr int kMaxStages = 2;
constexpr int kStageBytes = 16 * kChunkBytes;
constexpr size_t kSmemBudget = 112 * 1024;

__device__ unsigned int g_qmv_t5_timeouts = 0;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    return mbar_wait_for(bar, parity, kDrainWaitNs, &g_qmv_t5_timeouts);
}

struct T5Params {
    const __half *x;
    const uint8_t *w;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M, N, K, G;
    long long row_bytes;
    int tiles, chunks, S, Tc, Cs, NS;  // NS: stages per warp (1 or 2)
    uint32_t zero;  // always 0: keeps the magic constants in registers
};

template <int GS>
struct Geo {
    static constexpr int B = GS == 64 ? 13 : 26;    // bytes per group
    static constexpr int NG = GS == 64 ? 4 : 2;     // groups per thread slice
    static constexpr int NB = GS == 64 ? 2 : 1;     // bias MMAs per unit
    static constexpr int GPC = kChunkCodes / GS;    // groups per chunk
    // pair j (0..25) of a slice: byte a (group 2*beta) with byte a + B (group 2*beta+1)
    __host__ __device__ static constexpr int beta(int j) { return j / B; }
    __host__ __device__ static constexpr int byte_a(int j) { return 2 * B * (j / B) + j % B; }
};

__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

template <int GS, bool HAS_BIAS>
__global__ void __launch_bounds__(kThreads, 2) qmv_t5_kernel(const T5Params p)
{
    using Ge = Geo<GS>;
    constexpr int B = Ge::B;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(8) uint64_t fullbar[kWarps][kMaxStages];
    __shared__ __align__(8) uint64_t xbar;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int S = p.S;
    const int rank = S > 1 ? (int)cluster_ctarank() : 0;
    const int tile0 = (blockIdx.x / S) * p.Tc;
    const int ntile = min(p.Tc, p.tiles - tile0);
    const int c_lo = rank * p.Cs;
    const int ncl = max(0, min(p.Cs, p.chunks - c_lo));
    const int M = p.M;

    // shared memory: [lut][stages][Bs][SxB][raw x | accW accC]
    const int NS = p.NS;
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint8_t *stages = smem + 1024;
    // B fragments [Cs][M][4 slots][65 MMAs] (MMA index innermost: one base per
    // unit, immediate offsets per MMA)
    uint2 *Bs = reinterpret_cast<uint2 *>(stages + (size_t)kWarps * NS * kStageBytes);
    uint2 *SxB = Bs + (size_t)p.Cs * M * 4 * kMmas + 8 * 4 * kMmas;        // [Cs][NB][M][4] (+32 pad)
    uint8_t *region = reinterpret_cast<uint8_t *>(SxB + (size_t)p.Cs * Ge::NB * M * 4 + 32);
    __half *xr = reinterpret_cast<__half *>(region);                       // prologue only: [M][Cs*1024]
    float *accW = reinterpret_cast<float *>(region);                      // [warps][Tc][16][M]
    float *accC = accW + (size_t)kWarps * p.Tc * 16 * M;                   // [S][Tc][16][M]
    const int xs = p.Cs * kChunkCodes;  // raw x row stride (halves)
    // decode table: byte -> five trits at bits 0,2,4,6,8 (invalid bytes -> 0)
    {
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
    const uint32_t xb = smem_addr(&xbar);
    // the next kernel may launch now: it only prefetches weights until its
    // griddepcontrol.wait, which waits for this whole grid
    pdl_launch_dependents();
    if (tid == 0) mbar_init(xb, 1);
    if (lane == 0)
        for (int st = 0; st < NS; ++st) mbar_init(smem_addr(&fullbar[warp][st]), 1);

    pdl_wait();
    __syncthreads();

    // ---- raw x slice -> shared memory (bulk copies, one per row) --------------
    const long long k_lo = (long long)c_lo * kChunkCodes;
    const int slice_codes = ncl * kChunkCodes;  // K is a multiple of 1024 here
    if (tid == 0 && slice_codes > 0) {
        mbar_arrive_expect_tx(xb, (uint32_t)(M * slice_codes * 2));
        for (int m = 0; m < M; ++m)
            bulk_g2s(smem_addr(xr + (size_t)m * xs), p.x + (long long)m * p.K + k_lo, (uint32_t)(slice_codes * 2), xb);
    }
    bool x_ok = true;
    if (slice_codes > 0) x_ok = mbar_wait_bounded(xb, 0);
    const bool alive = __syncthreads_and(x_ok);
    if (!alive && tid == 0 && slice_codes > 0) mbar_wait_bounded(xb, 0);

    if (alive) {
        // B fragments: entry (cl, i, m, tt) = R0 (half2 2i), R1 (half2 2i+1) of
        // slot tt.  A thread owns fixed (i, tt) -- its four chunk-local code
        // offsets need only compile-time divisors -- and walks (cl, m).
        for (int it = tid; it < kMmas * 4; it += kThreads) {
            const int i = it >> 2, tt = it & 3;
            int kc[4];  // (slot, half) -> code within the chunk, -1 for a padding trit
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int sl = q >> 1, hi = q & 1;
                const int h = 2 * i + sl, j = h / 5, d = h % 5;
                const int o = Ge::byte_a(j) + hi * B;  // byte within the 52-byte slice
                const int grp = o / B, bg = o % B;      // slice-local group, byte in group
                const int within = 5 * bg + d;
                kc[q] = within < GS ? (Ge::NG * tt + grp) * GS + within : -1;
            }
            for (int cl = 0; cl < ncl; ++cl) {
                for (int m = 0; m < M; ++m) {
                    const uint16_t *src = reinterpret_cast<const uint16_t *>(xr) + (size_t)m * xs + cl * kChunkCodes;
                    uint32_t v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = kc[q] >= 0 ? src[kc[q]] : 0u;
                    Bs[((size_t)(cl * M + m) * 4 + tt) * kMmas + i] = make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
                }
            }
        }
        // bias MMA operands: groups gA = NG*tt + 2*nb, gB = gA + 1, (Sx_hi, Sx_lo) each
        const int sentries = ncl * Ge::NB * M * 4;
        for (int e = tid; e < sentries; e += kThreads) {
            const int tt = e & 3, m = (e >> 2) % M, nb = (e / (4 * M)) % Ge::NB, cl = e / (4 * M * Ge::NB);
            uint32_t r[2];
#pragma unroll
            for (int s_ = 0; s_ < 2; ++s_) {
                const int grp = Ge::NG * tt + 2 * nb + s_;
                const __half *src = xr + (size_t)m * xs + cl * kChunkCodes + grp * GS;
                float sx = 0.f;
                for (int q = 0; q < GS; q += 2) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(src + q));
                    sx += f.x;
                    sx += f.y;
                }
                const __half hi = __float2half_rn(sx);
                const __half lo = __float2half_rn(sx - __half2float(hi));
                r[s_] = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
            }
            SxB[e] = make_uint2(r[0], r[1]);
        }
    }
    __syncthreads();  // raw x consumed: its space becomes the accumulators
    for (int e = tid; e < kWarps * p.Tc * 16 * M; e += kThreads) accW[e] = 0.f;
    __syncthreads();
    if (S > 1) cluster_sync();

    // ---- per-warp stage ring --------------------------------------------------
    uint8_t *my_stages = stages + (size_t)warp * NS * kStageBytes;
    // one 208-byte bulk copy per weight row, issued by lanes 0..15
    auto issue = [&](int nidx, const UnitPos &pos) {
        if (pos.tl >= ntile) return;
        const int rowbase = (tile0 + pos.tl) * 16;
        const int nvalid = min(16, p.N - rowbase);
        const int st = NS == 2 ? (nidx & 1) : 0;
        const uint32_t bar = smem_addr(&fullbar[warp][st]);
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nvalid * kChunkBytes));
        __syncwarp();
        if (lane < nvalid) {
            const uint32_t dst = smem_addr(my_stages + st * kStageBytes + lane * kChunkBytes);
            const uint8_t *src = p.w + (long long)(rowbase + lane) * p.row_bytes +
                                 (long long)(c_lo + pos.cl) * kChunkBytes;
            bulk_g2s(dst, src, kChunkBytes, bar);
        }
    };

    uint32_t mg[5];
#pragma unroll
    for (int d = 0; d < 5; ++d) mg[d] = magic(2 * d) ^ p.zero;
    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
    auto flush = [&](int tl) {
        float *dst = accW + ((size_t)warp * p.Tc + tl) * 16 * M;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int col = 2 * t + (q & 1);
            if (col < M) dst[(g + 8 * (q >> 1)) * M + col] = (acc[0][q] + acc[1][q]) + (acc[2][q] + acc[3][q]);
            acc[0][q] = acc[1][q] = acc[2][q] = acc[3][q] = 0.f;
        }
    };

    if (alive && ncl > 0) {
        // prefetch distance = number of stages: unit n lives in stage n % NS,
        // and the stage is refilled with unit n + NS once unit n is in registers
        UnitPos ci, li;
        ci.start(warp, ncl);
        li = ci;
        for (int k = 0; k < NS; ++k) {
            issue(k, li);
            li.advance(ncl);
        }
        int cur_tile = ci.tl;
        for (int n = 0; ci.tl < ntile; ++n) {
            if (ci.tl != cur_tile) {
                flush(cur_tile);
                cur_tile = ci.tl;
            }
            const int st = NS == 2 ? (n & 1) : 0;
            const bool ok = mbar_wait_bounded(smem_addr(&fullbar[warp][st]), NS == 2 ? ((n >> 1) & 1) : (n & 1));
            if (!__all_sync(0xffffffffu, ok)) {
                // units n .. n+NS-1 may still have copies in flight: give each one
                // more bounded wait before leaving the loop
                UnitPos pend = ci;
                for (int k = 0; k < NS && pend.tl < ntile; ++k) {
                    const int nn = n + k;
                    mbar_wait_bounded(smem_addr(&fullbar[warp][NS == 2 ? (nn & 1) : 0]),
                                      NS == 2 ? ((nn >> 1) & 1) : (nn & 1));
                    pend.advance(ncl);
                }
                break;
            }
            // this lane's 52-byte slices of rows g and g+8
            const uint32_t *s0 = reinterpret_cast<const uint32_t *>(my_stages + st * kStageBytes + g * kChunkBytes + 52 * t);
            const uint32_t *s1 = s0 + 8 * kChunkBytes / 4;
            uint32_t wa[kSliceWords], wb[kSliceWords];
#pragma unroll
            for (int q = 0; q < kSliceWords; ++q) {
                wa[q] = s0[q];
                wb[q] = s1[q];
            }
            fence_proxy_async_smem();
            __syncwarp();
            issue(n + NS, li);
            li.advance(ncl);

            // scales (and biases) of this slice's groups, rows g and g+8
            const int rowg = (tile0 + ci.tl) * 16 + g;
            const int gslice = (c_lo + ci.cl) * Ge::GPC + Ge::NG * t;
            uint16_t sv[2][Ge::NG], bv[2][Ge::NG];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = rowg + 8 * rr;
                const bool rok = row < p.N;
                const __half *sp = p.scales + (long long)row * p.G + gslice;
                const __half *bp = (HAS_BIAS ? p.biases : p.scales) + (long long)row * p.G + gslice;
                uint32_t sw[2] = {0u, 0u}, bw[2] = {0u, 0u};
                if (Ge::NG == 4) {  // 4 halves, 8-byte aligned (G and the slice start are multiples of 4)
                    const uint2 a = ld_stream_v2_if(sp, rok);
                    sw[0] = a.x; sw[1] = a.y;
                    if (HAS_BIAS) { const uint2 b2 = ld_stream_v2_if(bp, rok); bw[0] = b2.x; bw[1] = b2.y; }
                } else {  // 2 halves, 4-byte aligned
                    sw[0] = ld_u32_if(sp, rok);
                    if (HAS_BIAS) bw[0] = ld_u32_if(bp, rok);
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
                        cst[rr][be][d] = hmul2(s2[rr][be], dup_half(__half_as_ushort(__float2half_rn(-(float)(1024 >> (2 * d))))));
                    fast = fast && fabsf(__half2float(__ushort_as_half(sv[rr][2 * be]))) < 63.f &&
                           fabsf(__half2float(__ushort_as_half(sv[rr][2 * be + 1]))) < 63.f;
                }
            const bool all_fast = __all_sync(0xffffffffu, fast);
            const uint2 *bq = Bs + ((size_t)(ci.cl * M + g) * 4 + t) * kMmas;

            auto pairs = [&](auto fast_tag) {
                constexpr bool kFast = decltype(fast_tag)::value;
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
                        const uint2 b = bq[i];
                        mma16816(acc[i & 3], A0[2 * q], A1[2 * q], A0[2 * q + 1], A1[2 * q + 1], b.x, b.y);
                    }
                }
            };
            if (all_fast) pairs(std::true_type{});
            else pairs(std::false_type{});
            // bias term
            const uint2 *sq = SxB + ((size_t)ci.cl * Ge::NB * M + g) * 4 + t;
#pragma unroll
            for (int nb = 0; nb < Ge::NB; ++nb) {
                const uint2 b = sq[(size_t)nb * M * 4];
                mma16816(acc[nb & 3], dup_half(bv[0][2 * nb]), dup_half(bv[1][2 * nb]), dup_half(bv[0][2 * nb + 1]),
                         dup_half(bv[1][2 * nb + 1]), b.x, b.y);
            }
            ci.advance(ncl);
        }
        if (cur_tile < ntile) flush(cur_tile);
    }
    __syncthreads();

    // ---- reduce: warps (fixed order), then cluster ranks (fixed order) ----------
    const int nout = ntile * 16 * M;
    for (int e = tid; e < nout; e += kThreads) {
        float v = 0.f;
        for (int w_ = 0; w_ < kWarps; ++w_) v += accW[(size_t)w_ * p.Tc * 16 * M + e];
        if (S > 1) st_cluster_f32(smem_addr(accC + (size_t)rank * p.Tc * 16 * M + e), 0, v);
        else accC[e] = v;
    }
    if (S > 1) {
        cluster_sync();
        if (rank != 0) return;
    } else {
        __syncthreads();
    }
    for (int e = tid; e < nout; e += kThreads) {
        const int tl = e / (16 * M), r = (e / M) % 16, m = e % M;
        const int n = (tile0 + tl) * 16 + r;
        if (n >= p.N) continue;
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += accC[(size_t)q * p.Tc * 16 * M + e];
        p.out[(size_t)m * p.N + n] = __float2half_rn(v);
    }
}

// ---- host side -----------------------------------------------------------------

struct Plan {
    int S, Tc, Cs, R, NS;
    size_t smem;
};

size_t smem_bytes(int gs, int M, int Cs, int Tc, int S, int NS)
{
    const int nb = gs == 64 ? 2 : 1;
    size_t b = 1024 + (size_t)kWarps * NS * kStageBytes;
    b += ((size_t)Cs * M * 4 * kMmas + 8 * 4 * kMmas) * sizeof(uint2);
    b += ((size_t)Cs * nb * M * 4 + 32) * sizeof(uint2);
    const size_t raw = (size_t)M * Cs * kChunkCodes * sizeof(__half);
    const size_t accs = (size_t)(kWarps + S) * Tc * 16 * M * sizeof(float);
    return b + (raw > accs ? raw : accs);
}

using OccFn = int (*)(int S, size_t smem);

bool make_plan(int gs, int M, int tiles, int chunks, int sms, OccFn occ, Plan &best)
{
    double best_cost = 1e30;
    bool found = false;
    // testing option: the stage count restricted to 1 or 2 (bqd_set_option)
    const int ns_only = opt_t5_stages();
    for (int NS = 2; NS >= 1; --NS) {
        if (ns_only && NS != ns_only) continue;
        for (int S = 1; S <= 8 && S <= chunks; ++S) {
            const int Cs = (chunks + S - 1) / S;
            if ((S - 1) * Cs >= chunks) continue;
            for (int Tc = 1; Tc <= kMaxTc; ++Tc) {
                const int R = (tiles + Tc - 1) / Tc;
                const size_t sm = smem_bytes(gs, M, Cs, Tc, S, NS);
                if (sm > kSmemBudget) continue;
                const int slots = S == 1 ? 2 * sms : occ(S, sm);
                if (slots <= 0) continue;
                const int waves = (R + slots - 1) / slots;
                const int per_warp = (Cs * Tc + kWarps - 1) / kWarps;
                // a unit is the bulk of the time; the prologue (x staging and
                // permute) costs ~0.15 unit per chunk and activation row plus a
                // copy round trip; a single stage exposes some copy latency
                const double cost = (double)waves * (per_warp * (NS == 2 ? 1.0 : 1.15) + 1.0 + 0.15 * Cs * M) + 0.01 * S;
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    best = Plan{S, Tc, Cs, R, NS, sm};
                    found = true;
                }
            }
        }
    }
    return found;
}

template <int GS, bool HAS_BIAS>
int cluster_slots(int S, size_t smem)
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
    auto kern = qmv_t5_kernel<GS, HAS_BIAS>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(kThreads);
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

template <int GS, bool HAS_BIAS>
int launch_t(const T5Params &p, const Plan &pl, cudaStream_t s)
{
    auto kern = qmv_t5_kernel<GS, HAS_BIAS>;
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.R * pl.S);
    cfg.blockDim = dim3(kThreads);
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
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
}

}  // namespace

int take_qmv_t5_timeouts(unsigned int *count)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmv_t5_timeouts, sizeof(v)) != cudaSuccess) return BQD_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_qmv_t5_timeouts, &zero, sizeof(zero)) != cudaSuccess) return BQD_ERR_CUDA;
    *count = v;
    return BQD_OK;
}

int launch_qmv_t5(const QmvArgs &a, cudaStream_t s)
{
    if (a.fmt != BQD_FMT_T5) return BQD_ERR_UNSUPPORTED;
    if (a.K % kChunkCodes != 0 || a.row_bytes % 16 != 0) return BQD_ERR_UNSUPPORTED;
    if (a.K > (int64_t)1 << 28 || a.N > (int64_t)1 << 28) return BQD_ERR_UNSUPPORTED;
    T5Params p;
    p.w = a.w; p.scales = a.scales; p.biases = a.biases; p.ratio = a.ratio;
    p.N = (int)a.N; p.K = (int)a.K; p.G = (int)a.G; p.row_bytes = a.row_bytes;
    p.tiles = (p.N + 15) / 16;
    p.chunks = p.K / kChunkCodes;
    p.zero = 0;
    const int sms = sm_count();
    const bool hb = a.biases != nullptr;
    for (int64_t m0 = 0; m0 < a.M; m0 += kMaxM) {
        const int M = (int)((a.M - m0) < kMaxM ? (a.M - m0) : kMaxM);
        OccFn occ = a.gs == 64 ? (hb ? cluster_slots<64, true> : cluster_slots<64, false>)
                               : (hb ? cluster_slots<128, true> : cluster_slots<128, false>);
        Plan pl;
        if (!make_plan(a.gs, M, p.tiles, p.chunks, sms, occ, pl)) return BQD_ERR_UNSUPPORTED;
        p.M = M;
        p.x = a.x + m0 * a.K;
        p.out = a.out + m0 * a.N;
        p.S = pl.S; p.Tc = pl.Tc; p.Cs = pl.Cs; p.NS = pl.NS;
        if (opt_debug_plan())
            fprintf(stderr, "bqd %s plan: N=%d K=%d M=%d gs=%d -> S=%d Tc=%d Cs=%d R=%d NS=%d grid=%d smem=%zu\n", "t5",
                    p.N, p.K, M, a.gs, pl.S, pl.Tc, pl.Cs, pl.R, pl.NS, pl.R * pl.S, pl.smem);
        int st;
        if (a.gs == 64) st = hb ? launch_t<64, true>(p, pl, s) : launch_t<64, false>(p, pl, s);
        else st = hb ? launch_t<128, true>(p, pl, s) : launch_t<128, false>(p, pl, s);
        if (st != BQD_OK) return st;
    }
    return BQD_OK;
}

}  // namespace bqd
