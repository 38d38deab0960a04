// Tensor-core decode QMV for 1-bit and 2-bit affine codes, M <= 8 rows of x.
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" -- §二.1 (qmv_fast:
// uint32-packed codes unpacked in registers, no floating-point weight matrix
// in memory), §二.2 (qmv_wide: one read of each weight byte serves all M rows;
// sym variant reads no bias tensor).
//
// y[m, n] = sum_k x[m,k] (s[n,g] q[n,k] + b[n,g])
//         = sum_k x[m,k] * A[n,k]  +  sum_g b[n,g] * Sx[m,g],
// with A = fp16(s*q) (exact for 1-bit; one rounding for 2-bit) and Sx the
// per-group sums of x.  Both sums run on the tensor cores (mma.sync
// m16n8k16 / m16n8k8, fp16 x fp16 -> fp32): weight rows are the MMA M
// dimension, the <= 8 activation rows the N dimension.  On CUDA cores the
// per-weight work is only the unpack: one LOP3 places a code into the
// mantissa of a "magic" fp16 whose exponent makes its value 2^(10-p) + q, and
// one HFMA2 with the constant -2^(10-p)*s turns that into s*q, for two codes
// at a time.  The bias term uses Sx split into an fp16 high part and an fp16
// remainder, so it carries no fp16 rounding of Sx.
//
// Work split: a "unit" is 16 weight rows x 256 codes.  A CTA owns a K-slice
// (Cs chunks of 256 codes) and Tc row tiles; its 8 warps take the slice's
// (tile, chunk) units round-robin.  x for the slice is staged once in shared
// memory in MMA B-fragment order.  When the K dimension is split over S > 1
// CTAs, the S CTAs form a thread-block cluster and the partial sums are
// reduced through distributed shared memory into the cluster's rank-0 CTA:
// no global scratch and no atomics, and the sum order is fixed, so results
// are bit-reproducible.  Weights are read with non-allocating 128/64-bit
// loads, two units ahead; the first units are requested before the
// programmatic-dependent-launch wait (weights never depend on the previous
// kernel).
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "bqd_internal.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

// Number of bounded device-side waits that expired (read by bqd_device_status).
__device__ unsigned int g_qmv_mma_timeouts = 0;

// Bounded wait: false (and the timeout counter bumped) if the phase never completes.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    return mbar_wait_for(bar, parity, kDrainWaitNs, &g_qmv_mma_timeouts);
}

constexpr int kThreads = kWarps * 32;
constexpr int kMaxM = 8;
constexpr int kMaxTc = 8;
constexpr int kCodesPerChunk = 256;  // per weight row, per unit
constexpr int kMmasPerChunk = 16;
constexpr size_t kSmemBudget = 112 * 1024;  // two CTAs per SM (228 KB, 1 KB reserved each)

struct Params {
    const __half *x;
    const uint8_t *w;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M, N, K, G, gs, lg_gs, gpc;
    uint32_t zero;  // always 0: makes the magic constants opaque so they stay in registers
    long long row_bytes;
    int tiles, chunks, S, Tc, Cs;
};

// ---- format traits -----------------------------------------------------------

template <int FMT> struct Fmt;

// 2-bit: 16 codes per word, a thread's slice of a unit is 4 words (16 B).
// Pair j (0..7) of a word = (code j, code j+8).  Codes 0..3 are read from
// w << 2 at mantissa bits 2,4,6,8; codes 4..7 from w >> 6 at the same bits.
template <> struct Fmt<BQD_FMT_AFFINE2> {
    static constexpr int kBits = 2, kCodesPerWord = 16, kWordsPerSlice = 4, kHalfOffset = 8;
    static constexpr int kNumPos = 4;
    // multiplier 2^(10-p) of the lowest code position (p=2) is 256: the
    // constant -256*s stays finite in fp16 for |s| <= 255
    static constexpr float kScaleLimit = 255.0f;
    __device__ static __forceinline__ float pos_mul(int i) { return (float)(256 >> (2 * i)); }
    __device__ static __forceinline__ void unpack_word(uint32_t w, uint32_t s2, const uint32_t (&c)[4],
                                                       const uint32_t (&mg)[4], uint32_t (&A)[8])
    {
        const uint32_t ua = w << 2, ub = w >> 6;
        A[0] = hfma2(and_or<0x00030003u << 2>(ua, mg[0]), s2, c[0]);
        A[1] = hfma2(and_or<0x00030003u << 4>(ua, mg[1]), s2, c[1]);
        A[2] = hfma2(and_or<0x00030003u << 6>(ua, mg[2]), s2, c[2]);
        A[3] = hfma2(and_or<0x00030003u << 8>(ua, mg[3]), s2, c[3]);
        A[4] = hfma2(and_or<0x00030003u << 2>(ub, mg[0]), s2, c[0]);
        A[5] = hfma2(and_or<0x00030003u << 4>(ub, mg[1]), s2, c[1]);
        A[6] = hfma2(and_or<0x00030003u << 6>(ub, mg[2]), s2, c[2]);
        A[7] = hfma2(and_or<0x00030003u << 8>(ub, mg[3]), s2, c[3]);
    }
    // magic for position index i (bits 2,4,6,8)
    __host__ __device__ static constexpr uint32_t magic_at(int i) { return magic(2 + 2 * i); }
    __device__ static __forceinline__ void unpack_word_exact(uint32_t w, uint32_t s2, uint32_t (&A)[8])
    {
        const uint32_t ua = w << 2, ub = w >> 6;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int p = 2 + 2 * (j & 3);
            const uint32_t u = j < 4 ? ua : ub;
            const uint32_t q = hsub2((u & (0x00030003u << p)) | magic(p), magic(p) & 0xfc00fc00u);
            A[j] = hmul2(q, s2);
        }
    }
};

// 1-bit: 32 codes per word, a thread's slice of a unit is 2 words (8 B).
// Pair j (0..15) of a word = (code j, code j+16).  Codes 0..4 come from
// w << 5, 5..9 from w, 10..14 from w >> 5 (mantissa bits 5..9), code 15 from
// w >> 6 (bit 9).
template <> struct Fmt<BQD_FMT_AFFINE1> {
    static constexpr int kBits = 1, kCodesPerWord = 32, kWordsPerSlice = 2, kHalfOffset = 16;
    static constexpr int kNumPos = 5;
    // lowest position p=5: multiplier 32, finite for |s| <= 2047
    static constexpr float kScaleLimit = 2047.0f;
    __device__ static __forceinline__ float pos_mul(int i) { return (float)(32 >> i); }
    __device__ static __forceinline__ void unpack_word(uint32_t w, uint32_t s2, const uint32_t (&c)[5],
                                                       const uint32_t (&mg)[5], uint32_t (&A)[16])
    {
        const uint32_t u0 = w << 5, u2 = w >> 5, u3 = w >> 6;
        A[0] = hfma2(and_or<0x00010001u << 5>(u0, mg[0]), s2, c[0]);
        A[1] = hfma2(and_or<0x00010001u << 6>(u0, mg[1]), s2, c[1]);
        A[2] = hfma2(and_or<0x00010001u << 7>(u0, mg[2]), s2, c[2]);
        A[3] = hfma2(and_or<0x00010001u << 8>(u0, mg[3]), s2, c[3]);
        A[4] = hfma2(and_or<0x00010001u << 9>(u0, mg[4]), s2, c[4]);
        A[5] = hfma2(and_or<0x00010001u << 5>(w, mg[0]), s2, c[0]);
        A[6] = hfma2(and_or<0x00010001u << 6>(w, mg[1]), s2, c[1]);
        A[7] = hfma2(and_or<0x00010001u << 7>(w, mg[2]), s2, c[2]);
        A[8] = hfma2(and_or<0x00010001u << 8>(w, mg[3]), s2, c[3]);
        A[9] = hfma2(and_or<0x00010001u << 9>(w, mg[4]), s2, c[4]);
        A[10] = hfma2(and_or<0x00010001u << 5>(u2, mg[0]), s2, c[0]);
        A[11] = hfma2(and_or<0x00010001u << 6>(u2, mg[1]), s2, c[1]);
        A[12] = hfma2(and_or<0x00010001u << 7>(u2, mg[2]), s2, c[2]);
        A[13] = hfma2(and_or<0x00010001u << 8>(u2, mg[3]), s2, c[3]);
        A[14] = hfma2(and_or<0x00010001u << 9>(u2, mg[4]), s2, c[4]);
        A[15] = hfma2(and_or<0x00010001u << 9>(u3, mg[4]), s2, c[4]);
    }
    // magic for position index i (bits 5..9)
    __host__ __device__ static constexpr uint32_t magic_at(int i) { return magic(5 + i); }
    __device__ static __forceinline__ void unpack_word_exact(uint32_t w, uint32_t s2, uint32_t (&A)[16])
    {
        const uint32_t u0 = w << 5, u1 = w, u2 = w >> 5, u3 = w >> 6;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int p = j == 15 ? 9 : 5 + (j % 5);
            const uint32_t u = j < 5 ? u0 : (j < 10 ? u1 : (j < 15 ? u2 : u3));
            const uint32_t q = hsub2((u & (0x00010001u << p)) | magic(p), magic(p) & 0xfc00fc00u);
            A[j] = hmul2(q, s2);
        }
    }
};

// Per-thread data of one unit.
struct UnitData {
    uint4 w0, w1;     // slice of row g / row g+8 (1-bit uses .x, .y)
    uint16_t s0, s1;  // scale of the slice's group, rows g / g+8
    uint16_t b0, b1;  // bias (sym: scale) of the bias-MMA group, rows g / g+8
};

// Global addresses of one warp's next unit to load, advanced incrementally.
template <int FMT, bool HAS_BIAS>
struct LoadIter {
    static constexpr int SB = Fmt<FMT>::kWordsPerSlice * 4;  // slice bytes per thread
    UnitPos pos;
    const uint8_t *wp;  // weight slice, row g
    const __half *sp;   // scale of the slice's group, row g
    const __half *bp;   // bias (sym: scale) of the bias-MMA group, row g
    int rowg;           // global index of row g
    int byte_off;       // slice byte offset within the row
    int gb;             // bias-MMA group index

    __device__ __forceinline__ void init(const Params &p, int tile0, int c_lo, int ncl, int warp, int g, int t)
    {
        pos.start(warp, ncl);
        const int c = c_lo + pos.cl;
        rowg = (tile0 + pos.tl) * 16 + g;
        byte_off = c * 4 * SB + t * SB;
        gb = c * p.gpc + t;
        const int gsl = (int)(((long long)byte_off * (8 / Fmt<FMT>::kBits)) >> p.lg_gs);
        wp = p.w + (long long)rowg * p.row_bytes + byte_off;
        sp = p.scales + (long long)rowg * p.G + gsl;
        bp = (HAS_BIAS ? p.biases : p.scales) + (long long)rowg * p.G + gb;
    }

    __device__ __forceinline__ void advance(const Params &p, int ncl)
    {
        const int crossed = pos.advance(ncl);
        if (crossed == 0) {  // common case: next chunk of the same row tile
            wp += kWarps * 4 * SB;
            sp += kWarps * p.gpc;
            bp += kWarps * p.gpc;
            byte_off += kWarps * 4 * SB;
            gb += kWarps * p.gpc;
            return;
        }
        const int dchunk = kWarps - crossed * ncl;  // net chunk step
        wp += (long long)crossed * 16 * p.row_bytes + (long long)dchunk * 4 * SB;
        sp += (long long)crossed * 16 * p.G + dchunk * p.gpc;
        bp += (long long)crossed * 16 * p.G + dchunk * p.gpc;
        rowg += crossed * 16;
        byte_off += dchunk * 4 * SB;
        gb += dchunk * p.gpc;
    }

    __device__ __forceinline__ void load(const Params &p, int ntile, int t, UnitData &d) const
    {
        const bool live = pos.tl < ntile;
        const long long r8 = 8 * p.row_bytes;
        const int g8 = 8 * p.G;
        // warp-uniform: the whole unit lies inside the matrix (no tail row
        // tile, no tail chunk): plain loads, no predicates
        const bool interior = live && rowg - (rowg & 15) + 16 <= p.N &&
                              byte_off - t * SB + 4 * SB <= p.row_bytes && gb - t + p.gpc <= p.G;
        if (__all_sync(0xffffffffu, interior)) {
            if (SB == 16) {
                d.w0 = ld_stream_v4(wp);
                d.w1 = ld_stream_v4(wp + r8);
            } else {
                const uint2 a = ld_stream_v2(wp), b = ld_stream_v2(wp + r8);
                d.w0 = make_uint4(a.x, a.y, 0, 0);
                d.w1 = make_uint4(b.x, b.y, 0, 0);
            }
            d.s0 = ld_u16(sp);
            d.s1 = ld_u16(sp + g8);
            const bool gb_ok = t < p.gpc;
            d.b0 = ld_u16_if(bp, gb_ok);
            d.b1 = ld_u16_if(bp + g8, gb_ok);
            return;
        }
        const bool ok0 = live && byte_off < p.row_bytes && rowg < p.N;
        const bool ok1 = live && byte_off < p.row_bytes && rowg + 8 < p.N;
        const bool gb_ok = live && t < p.gpc && gb < p.G;
        if (SB == 16) {
            d.w0 = ld_stream_v4_if(wp, ok0);
            d.w1 = ld_stream_v4_if(wp + r8, ok1);
        } else {
            const uint2 a = ld_stream_v2_if(wp, ok0), b = ld_stream_v2_if(wp + r8, ok1);
            d.w0 = make_uint4(a.x, a.y, 0, 0);
            d.w1 = make_uint4(b.x, b.y, 0, 0);
        }
        d.s0 = ld_u16_if(sp, ok0);
        d.s1 = ld_u16_if(sp + g8, ok1);
        d.b0 = ld_u16_if(bp, gb_ok && rowg < p.N);
        d.b1 = ld_u16_if(bp + g8, gb_ok && rowg + 8 < p.N);
    }
};

// Constants -2^(10-p)*s (fp16x2) of one row's slice; false when |s| is too
// large for them (the exact, slower unpack is then used for the unit).
template <int FMT>
__device__ __forceinline__ bool row_constants(uint16_t s, uint32_t &s2, uint32_t (&c)[Fmt<FMT>::kNumPos])
{
    using F = Fmt<FMT>;
    s2 = dup_half(s);
#pragma unroll
    for (int i = 0; i < F::kNumPos; ++i)
        c[i] = hmul2(s2, dup_half(__half_as_ushort(__float2half_rn(-F::pos_mul(i)))));
    return fabsf(__half2float(__ushort_as_half(s))) <= F::kScaleLimit;
}

// B fragments in shared memory: [chunk][mma][MP columns][4 slots] uint2.
// Lanes whose column g >= MP read column g mod MP: those output columns are
// never stored.
template <int FMT, bool HAS_BIAS, int MP>
__device__ __forceinline__ void compute_unit(const Params &p, const UnitData &d, int cl, int bl,
                                             const uint2 *__restrict__ Bs, const uint32_t *__restrict__ SxB,
                                             const uint32_t (&mg)[Fmt<FMT>::kNumPos], float (&acc)[4][4])
{
    using F = Fmt<FMT>;
    constexpr int WPS = F::kWordsPerSlice;
    constexpr int PPW = 32 / F::kBits / 2;  // pairs per word
    uint32_t s20, s21, c0[F::kNumPos], c1[F::kNumPos];
    const bool fast = row_constants<FMT>(d.s0, s20, c0) & row_constants<FMT>(d.s1, s21, c1);
    const uint32_t w0[4] = {d.w0.x, d.w0.y, d.w0.z, d.w0.w};
    const uint32_t w1[4] = {d.w1.x, d.w1.y, d.w1.z, d.w1.w};
    const uint2 *bq = Bs + cl * (kMmasPerChunk * MP * 4) + bl;
    if (__all_sync(0xffffffffu, fast)) {
#pragma unroll
        for (int u = 0; u < WPS; ++u) {
            uint32_t A0[PPW], A1[PPW];
            F::unpack_word(w0[u], s20, c0, mg, A0);
            F::unpack_word(w1[u], s21, c1, mg, A1);
#pragma unroll
            for (int jj = 0; jj < PPW / 2; ++jj) {
                const int i = u * (PPW / 2) + jj;
                const uint2 b = bq[i * MP * 4];
                mma16816(acc[i & 3], A0[2 * jj], A1[2 * jj], A0[2 * jj + 1], A1[2 * jj + 1], b.x, b.y);
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < WPS; ++u) {
            uint32_t A0[PPW], A1[PPW];
            F::unpack_word_exact(w0[u], s20, A0);
            F::unpack_word_exact(w1[u], s21, A1);
#pragma unroll
            for (int jj = 0; jj < PPW / 2; ++jj) {
                const int i = u * (PPW / 2) + jj;
                const uint2 b = bq[i * MP * 4];
                mma16816(acc[i & 3], A0[2 * jj], A1[2 * jj], A0[2 * jj + 1], A1[2 * jj + 1], b.x, b.y);
            }
        }
    }
    // bias term: A = b (duplicated), B = (Sx_hi, Sx_lo) of the same group
    uint16_t b0 = d.b0, b1 = d.b1;
    if (!HAS_BIAS) {
        b0 = __half_as_ushort(sym_bias(__ushort_as_half(d.b0), p.ratio));
        b1 = __half_as_ushort(sym_bias(__ushort_as_half(d.b1), p.ratio));
    }
    mma1688(acc[3], dup_half(b0), dup_half(b1), SxB[cl * MP * 4 + bl]);
}

template <int FMT, bool HAS_BIAS, int MP>
__global__ void __launch_bounds__(kThreads, 2) qmv_mma_kernel(const Params p)
{
    using F = Fmt<FMT>;
    constexpr int CPW = F::kCodesPerWord;
    constexpr int HO = F::kHalfOffset;
    constexpr int WPS = F::kWordsPerSlice;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(8) uint64_t xbar;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int bl = (g & (MP - 1)) * 4 + t;  // this lane's B column/slot
    const int S = p.S;
    const int rank = S > 1 ? (int)cluster_ctarank() : 0;
    const int tile0 = (blockIdx.x / S) * p.Tc;
    const int ntile = min(p.Tc, p.tiles - tile0);
    const int c_lo = rank * p.Cs;
    const int ncl = max(0, min(p.Cs, p.chunks - c_lo));
    const int M = p.M;

    // shared memory carve-up (sizes must match smem_bytes())
    const int RS = p.Cs * kCodesPerChunk + 8;  // raw x row stride (halves): 16 mod 128 bytes
    uint2 *Bs = reinterpret_cast<uint2 *>(smem);                                       // [Cs][16][MP][4]
    uint32_t *SxB = reinterpret_cast<uint32_t *>(Bs + (size_t)p.Cs * kMmasPerChunk * MP * 4);  // [Cs][MP][4]
    uint8_t *region = reinterpret_cast<uint8_t *>(SxB + (size_t)p.Cs * MP * 4);
    __half *xr = reinterpret_cast<__half *>(region);   // [M][RS], prologue only
    float *accW = reinterpret_cast<float *>(region);  // [warps][Tc][16][8], after the prologue
    float *accC = accW + (size_t)kWarps * p.Tc * 128;  // [S][Tc][16][8]
    const uint32_t bar = smem_addr(&xbar);
    // the next kernel may launch now: it only prefetches weights until its
    // griddepcontrol.wait, which waits for this whole grid
    pdl_launch_dependents();
    if (tid == 0) mbar_init(bar, 1);

    // ---- weights of the first three units: independent of the previous kernel --
    const bool any = ncl > 0;
    UnitData d0, d1, d2;
    LoadIter<FMT, HAS_BIAS> li;
    UnitPos ci;
    if (any) {
        li.init(p, tile0, c_lo, ncl, warp, g, t);
        ci = li.pos;
        li.load(p, ntile, t, d0);
        li.advance(p, ncl);
        li.load(p, ntile, t, d1);
        li.advance(p, ncl);
        li.load(p, ntile, t, d2);
        li.advance(p, ncl);
    }

    pdl_wait();

    // ---- raw x slice -> shared memory: one bulk (TMA) copy per row -------------
    const long long k_lo = (long long)c_lo * kCodesPerChunk;
    const int slice_codes = (int)max(0LL, min((long long)ncl * kCodesPerChunk, (long long)p.K - k_lo));
    __syncthreads();  // barrier initialised before anyone waits on it
    if (tid == 0 && slice_codes > 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)(M * slice_codes * 2));
        for (int m = 0; m < M; ++m)
            bulk_g2s(smem_addr(xr + (size_t)m * RS), p.x + (long long)m * p.K + k_lo, (uint32_t)(slice_codes * 2), bar);
    }
    bool x_ok = true;
    if (slice_codes > 0) x_ok = mbar_wait_bounded(bar, 0);
    // A CTA whose copy never completed gives it one more bounded wait, then does
    // no work but still passes every barrier (its cluster peers wait on them);
    // the timeout is reported through bqd_device_status().
    const bool alive = __syncthreads_and(x_ok);
    if (!alive && tid == 0 && slice_codes > 0) mbar_wait_bounded(bar, 0);

    // ---- permute to B-fragment order; lane = (column m, slot t_) ---------------
    if (alive) {
        const int m = lane >> 2, t_ = lane & 3;
        for (int cu = warp; m < MP && cu < ncl * WPS; cu += kWarps) {
            const int cl = cu / WPS, u = cu % WPS;
            const int lw = cl * 4 * WPS + t_ * WPS + u;  // word within the slice
            uint32_t v[CPW / 2];
            const bool ok = m < M && lw * CPW < slice_codes;
#pragma unroll
            for (int q = 0; q < CPW / 8; ++q) {
                uint4 x4 = make_uint4(0, 0, 0, 0);
                if (ok) x4 = *reinterpret_cast<const uint4 *>(xr + (size_t)m * RS + lw * CPW + 8 * q);
                v[4 * q] = x4.x; v[4 * q + 1] = x4.y; v[4 * q + 2] = x4.z; v[4 * q + 3] = x4.w;
            }
#pragma unroll
            for (int jj = 0; jj < HO / 2; ++jj) {
                // R0 = (x[2jj], x[2jj+HO]), R1 = (x[2jj+1], x[2jj+HO+1])
                const uint32_t lo = v[jj], hi = v[jj + HO / 2];
                uint2 b;
                b.x = __byte_perm(lo, hi, 0x5410);
                b.y = __byte_perm(lo, hi, 0x7632);
                Bs[((size_t)cl * kMmasPerChunk + u * (HO / 2) + jj) * (MP * 4) + m * 4 + t_] = b;
            }
        }
        // group sums Sx in a fixed order, split into fp16 high part + remainder
        for (int e = tid; e < ncl * MP * 4; e += kThreads) {
            const int cl = e / (MP * 4), mm = (e / 4) % MP, tt = e % 4;
            uint32_t packed = 0;
            const int k0 = cl * kCodesPerChunk + tt * p.gs;
            if (tt < p.gpc && mm < M && k0 < slice_codes) {
                const __half *src = xr + (size_t)mm * RS + k0;
                float sx = 0.f;
                for (int q = 0; q < p.gs; q += 8) {
                    const uint4 x4 = *reinterpret_cast<const uint4 *>(src + q);
                    const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&xw[h]));
                        sx += f.x;
                        sx += f.y;
                    }
                }
                const __half hi = __float2half_rn(sx);
                const __half lo = __float2half_rn(sx - __half2float(hi));
                packed = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
            }
            SxB[e] = packed;
        }
    }
    __syncthreads();  // raw x no longer needed: its space becomes the accumulators
    for (int e = tid; e < kWarps * p.Tc * 128; e += kThreads) accW[e] = 0.f;
    __syncthreads();
    if (S > 1) cluster_sync();  // rank 0's accumulators exist before anyone writes them

    // ---- main loop: two units in flight while one is computed -------------------
    uint32_t mg[F::kNumPos];
#pragma unroll
    for (int i = 0; i < F::kNumPos; ++i) mg[i] = F::magic_at(i) ^ p.zero;
    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
    int cur_tile = ci.tl;
    auto flush = [&](int tl) {
        float *dst = accW + ((size_t)warp * p.Tc + tl) * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float v = (acc[0][q] + acc[1][q]) + (acc[2][q] + acc[3][q]);
            dst[(g + 8 * (q >> 1)) * 8 + 2 * t + (q & 1)] = v;
            acc[0][q] = acc[1][q] = acc[2][q] = acc[3][q] = 0.f;
        }
    };
    auto step = [&](UnitData &d) {
        if (ci.tl != cur_tile) {
            flush(cur_tile);
            cur_tile = ci.tl;
        }
        compute_unit<FMT, HAS_BIAS, MP>(p, d, ci.cl, bl, Bs, SxB, mg, acc);
        ci.advance(ncl);
        li.load(p, ntile, t, d);
        li.advance(p, ncl);
    };
    if (any && alive) {
        while (ci.tl < ntile) {
            step(d0);
            if (ci.tl >= ntile) break;
            step(d1);
            if (ci.tl >= ntile) break;
            step(d2);
        }
        if (cur_tile < ntile) flush(cur_tile);
    }
    __syncthreads();

    // ---- reduce: warps (fixed order), then cluster ranks (fixed order) ----------
    const int nout = ntile * 128;
    for (int e = tid; e < nout; e += kThreads) {
        float v = 0.f;
        for (int w_ = 0; w_ < kWarps; ++w_) v += accW[(size_t)w_ * p.Tc * 128 + e];
        if (S > 1) st_cluster_f32(smem_addr(accC + (size_t)rank * p.Tc * 128 + e), 0, v);
        else accC[e] = v;
    }
    if (S > 1) {
        cluster_sync();
        if (rank != 0) return;
    } else {
        __syncthreads();
    }
    for (int e = tid; e < ntile * 16 * M; e += kThreads) {
        const int tl = e / (16 * M), r = (e / M) % 16, m = e % M;
        const int n = (tile0 + tl) * 16 + r;
        if (n >= p.N) continue;
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += accC[((size_t)q * p.Tc + tl) * 128 + r * 8 + m];
        p.out[(size_t)m * p.N + n] = __float2half_rn(v);
    }
}

// ---- host side -----------------------------------------------------------------

struct Plan {
    int S, Tc, Cs, R, MP;
    size_t smem;
};

size_t smem_bytes(int MP, int M, int Cs, int Tc, int S)
{
    size_t b = (size_t)Cs * kMmasPerChunk * MP * 4 * sizeof(uint2);  // Bs
    b += (size_t)Cs * MP * 4 * sizeof(uint32_t);                      // SxB
    const size_t raw = (size_t)M * (Cs * kCodesPerChunk + 8) * sizeof(__half);
    const size_t accs = (size_t)(kWarps + S) * Tc * 128 * sizeof(float);
    return b + (raw > accs ? raw : accs);
}

// Largest number of co-resident clusters of size S for a kernel using `smem`
// bytes per CTA (queried once per configuration; 0 when unavailable).
using OccFn = int (*)(int S, size_t smem);

bool make_plan(int M, int tiles, int chunks, int sms, OccFn occ, Plan &best)
{
    double best_cost = 1e30;
    bool found = false;
    const int MP = M <= 4 ? 4 : 8;
    for (int S = 1; S <= 8 && S <= chunks; ++S) {
        const int Cs = (chunks + S - 1) / S;
        if ((S - 1) * Cs >= chunks) continue;
        for (int Tc = 1; Tc <= kMaxTc; ++Tc) {
            const int R = (tiles + Tc - 1) / Tc;
            const size_t sm = smem_bytes(MP, M, Cs, Tc, S);
            if (sm > kSmemBudget) continue;
            // co-resident clusters (S CTAs each); S = 1: two CTAs per SM
            int slots = S == 1 ? 2 * sms : occ(S, sm);
            if (slots <= 0) continue;
            const int waves = (R + slots - 1) / slots;
            const int per_warp = (Cs * Tc + kWarps - 1) / kWarps;
            // time ~ waves x (units per warp + a prologue worth ~3 units)
            const double cost = (double)waves * (per_warp + 3) + 0.01 * S;
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best = Plan{S, Tc, Cs, R, MP, sm};
                found = true;
            }
        }
    }
    return found;
}

template <int FMT, bool HAS_BIAS, int MP>
int launch_t(const Params &p, const Plan &pl, cudaStream_t s)
{
    auto kern = qmv_mma_kernel<FMT, HAS_BIAS, MP>;
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
}

// Co-resident clusters of S CTAs of one kernel instantiation (cached).
template <int FMT, bool HAS_BIAS, int MP>
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
    auto kern = qmv_mma_kernel<FMT, HAS_BIAS, MP>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
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

template <int FMT>
int launch_fmt(const Params &p, const Plan &pl, bool has_bias, cudaStream_t s)
{
    if (pl.MP == 4)
        return has_bias ? launch_t<FMT, true, 4>(p, pl, s) : launch_t<FMT, false, 4>(p, pl, s);
    return has_bias ? launch_t<FMT, true, 8>(p, pl, s) : launch_t<FMT, false, 8>(p, pl, s);
}

template <int FMT>
OccFn occ_fn(bool has_bias, int MP)
{
    if (MP == 4) return has_bias ? cluster_slots<FMT, true, 4> : cluster_slots<FMT, false, 4>;
    return has_bias ? cluster_slots<FMT, true, 8> : cluster_slots<FMT, false, 8>;
}

}  // namespace

int take_qmv_mma_timeouts(unsigned int *count)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmv_mma_timeouts, sizeof(v)) != cudaSuccess) return BQD_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_qmv_mma_timeouts, &zero, sizeof(zero)) != cudaSuccess) return BQD_ERR_CUDA;
    *count = v;
    return BQD_OK;
}

int launch_qmv_mma(const QmvArgs &a, cudaStream_t s)
{
    if (a.fmt != BQD_FMT_AFFINE1 && a.fmt != BQD_FMT_AFFINE2) return BQD_ERR_UNSUPPORTED;
    if (a.K > (int64_t)1 << 28 || a.N > (int64_t)1 << 28) return BQD_ERR_UNSUPPORTED;
    Params p;
    p.w = a.w; p.scales = a.scales; p.biases = a.biases; p.ratio = a.ratio;
    p.N = (int)a.N; p.K = (int)a.K; p.G = (int)a.G; p.gs = a.gs; p.lg_gs = a.gs == 64 ? 6 : 7;
    p.gpc = kCodesPerChunk / a.gs;
    p.row_bytes = a.row_bytes;
    p.zero = 0;
    p.tiles = (p.N + 15) / 16;
    p.chunks = (p.K + kCodesPerChunk - 1) / kCodesPerChunk;
    const int sms = sm_count();
    for (int64_t m0 = 0; m0 < a.M; m0 += kMaxM) {
        const int M = (int)((a.M - m0) < kMaxM ? (a.M - m0) : kMaxM);
        Plan pl;
        const int MP = M <= 4 ? 4 : 8;
        const bool hb = a.biases != nullptr;
        const OccFn occ = a.fmt == BQD_FMT_AFFINE2 ? occ_fn<BQD_FMT_AFFINE2>(hb, MP) : occ_fn<BQD_FMT_AFFINE1>(hb, MP);
        if (!make_plan(M, p.tiles, p.chunks, sms, occ, pl)) return BQD_ERR_UNSUPPORTED;
        p.M = M;
        p.x = a.x + m0 * a.K;
        p.out = a.out + m0 * a.N;
        p.S = pl.S; p.Tc = pl.Tc; p.Cs = pl.Cs;
        if (opt_debug_plan())
            fprintf(stderr, "bqd %s plan: N=%d K=%d M=%d gs=%d -> S=%d Tc=%d Cs=%d R=%d grid=%d smem=%zu\n", "mma",
                    p.N, p.K, M, a.gs, pl.S, pl.Tc, pl.Cs, pl.R, pl.R * pl.S, pl.smem);
        const int st = a.fmt == BQD_FMT_AFFINE2 ? launch_fmt<BQD_FMT_AFFINE2>(p, pl, a.biases != nullptr, s)
                                                : launch_fmt<BQD_FMT_AFFINE1>(p, pl, a.biases != nullptr, s);
        if (st != BQD_OK) return st;
    }
    return BQD_OK;
}

}  // namespace bqd
