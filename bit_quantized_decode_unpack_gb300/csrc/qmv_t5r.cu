// Tensor-core decode QMV for t5 ternary weights fed by TMA into a shared-memory
// ring (M <= 8 activation rows per pass, K a multiple of 1024).
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" -- §二.3 (t5:
// trits {0,1,2}, five per uint8, 13 bytes per 64-weight group / 26 per
// 128-weight group), §二.2 (one read of every weight byte serves all M rows;
// the sym variant rebuilds the bias from the scale).
//
//   y[m,n] = sum_g s[n,g] * sum_{k in g} x[m,k] t[n,k]  +  sum_g b[n,g] Sx[m,g]
//
// Decode without a table.  Two bytes a, b of one group go into the halves of
// an fp16x2 as 1024 + v (one PRMT against the exponent byte 0x64).  Integer
// division by three is one fused fp16 multiply-add: for Q = 1024 + q with
// q <= 242, fma(Q, fp16(1/3), 682.5) rounds to exactly 1024 + floor(q/3)
// (checked for every byte value).  So
//     Q0 = V,  Q(d+1) = fma(Qd, 1/3, 682.5),  A_d = fma(Q(d+1), -3, Qd) = t_d - 2048
// for d < 4, and A_4 = Q4 = 1024 + t_4: eight HFMA2 give the five digits of
// both bytes exactly.  A group's byte without a partner pairs two of its own
// digits: its high half starts one division ahead.
//
// Layout of the codes on the MMA (mma.sync m16n8k16, fp32 accumulation,
// weight rows = MMA rows): thread t of a quad takes codes [256t, 256t+256)
// of a row's 1024-code chunk (four whole groups of 64, or two of 128), one
// group ("period") at a time; its k-slots of MMA i of a period hold items 2i
// and 2i+1 of that group (item = the two codes of one A register).  Two ways
// to apply the scale:
//  * column split (passes of M <= 2 x rows): B column 2t+e holds x row e at
//    thread t's k-slots and zeros at the other threads' slots, so D[n][2t+e]
//    sums thread t's current group alone, and s (D - Cx) + b Sx adds it in
//    fp32.  Cx (the offsets' dot product) and Sx (the group sum of x) come
//    from the same MMA sequence over a constant A (row 0 ones, row 1 the
//    offsets), run once per chunk by the producer: a row whose trits in a
//    group are all zero gives D == Cx bit for bit.  No weight is scaled.
//  * scaled (M >= 3): fma(A, s, 2048 s) (or -1024 s for digit 4) gives
//    fp16(s t) exactly while |s| < 32 (a warp with larger scales takes the
//    exact (A + 2048) s form), the B columns are the x rows, and one MMA per
//    A fragment serves all M <= 8 rows.  The bias term is one MMA per two
//    groups per chunk, against the group sums of x split into an fp16 high
//    part and remainder.
//
// CTA: NW consumer warps (warp w owns weight rows n0+16w .. +15) and two
// producer warps, which prepare alternate chunks (one alone could not keep up
// with the consumers from two x rows on); NW = 8 (128 rows, two CTAs per SM)
// for passes of up to five x rows, 16 (256 rows, one CTA per SM) for larger
// passes.  Per ring stage (one 1024-code chunk of the CTA's rows) a producer
// issues the 2-D TMA copies of the weights [rows][208 B], the scales and the
// biases, then builds the B fragments from the chunk of x (16-byte copies
// through the load/store path into its own buffer, requested once its previous
// chunk's fragments are built; each pass of the warp gathers from one x row)
// and the sums above.  Weights, scales and
// biases are requested before the programmatic-dependent-launch wait.  K is
// split over the S CTAs of a cluster.  The partial sums are reduce-scattered
// through distributed shared memory, each rank adding its slice of rows in
// rank order (deterministic, no global scratch).  Every mbarrier wait is
// bounded.  An expiry is counted for bqd_device_status.
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

constexpr int kCodesR = 1024;                  // codes per row per stage
constexpr int kBytesR = 208;                   // t5 bytes per row per stage
constexpr int kSliceR = 52;                    // bytes of one thread's slice of a row chunk
constexpr int kMmasR = 64;                     // MMAs per 16 rows per chunk
constexpr int kPairsR = kMmasR / 2;            // B entries of two MMAs each, per slot and x row
constexpr int kMaxMR = 8;                      // x rows per pass (the MMA's N)
constexpr int kMaxStagesR = 4;
constexpr int kMaxSplitR = 16;

// CTA shape: NW consumer warps of 16 weight rows each plus two producer warps
// (alternate chunks): NW = 8 (128 rows, two CTAs per SM) or NW = 16 (256 rows,
// one CTA per SM).
constexpr int kProdR = 2;
template <int NW>
struct Cta {
    static constexpr int kThreads = (NW + kProdR) * 32;
    static constexpr int kRows = 16 * NW;
    static constexpr int kPerSM = NW == 16 ? 1 : 2;
    static constexpr size_t kSmemBudget = NW == 16 ? 224 * 1024 : 110 * 1024;  // dynamic (static ~3 KB)
};

struct T5RParams {
    const uint8_t *w;  // host side only (the weight tensor map)
    const __half *x;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M;     // x rows per pass (the staging and fragment layouts)
    int Mtot;  // x rows of the call; pass blockIdx.y takes rows M*y .. M*y+M-1
    int N, K, G, chunks, S, Cs, stages, RS;
    uint32_t stage_bytes;
    uint32_t zero;  // always 0: keeps the fp16 constants opaque (in registers)
    unsigned long long wait_ns;  // limit of the pipeline waits
};

// ---- the items of a group ----------------------------------------------------------
//
// A group of GS codes is B bytes (byte c holds codes 5c .. 5c+4, digit d = code
// 5c + d).  It is cut into GS/2 "items", each the two halves of one A
// register:
//   * items 5j .. 5j+4: bytes 2j and 2j+1, digit d = item - 5j;
//   * gs=64: items 30, 31 take byte 12 (four real codes, its digit 4 is
//     padding) as digit pairs (0,1) and (2,3) of the byte itself;
//   * gs=128: items 60..62 take bytes 24 and 25, digits 0..2 (digits 3, 4
//     of byte 25 are padding); item 63 takes digits (3,4) of byte 24.
// MMA i of a group period uses items 2i (k-slots 2t, 2t+1) and 2i+1 (slots
// 2t+8, 2t+9).
template <int GS>
struct T5G {
    static constexpr int B = GS == 64 ? 13 : 26;   // bytes per group
    static constexpr int NG = kCodesR / 4 / GS;    // groups per thread slice: 4 or 2
    static constexpr int NB = NG / 2;              // bias MMAs per chunk (two groups each)
    static constexpr int GPC = kCodesR / GS;       // groups per chunk
    static constexpr int MPG = GS / 4;             // MMAs per group period (a thread fills 4 k-slots of each)
    static constexpr int NP = GS == 64 ? 6 : 12;   // full byte pairs (five items each)
    __host__ __device__ static constexpr int byte_a(int u) { return u < 5 * NP ? 2 * (u / 5) : (GS == 64 ? 12 : 24); }
    // the partner byte of item u, or -1 when the item pairs two digits of byte_a
    __host__ __device__ static constexpr int byte_b(int u)
    {
        return u < 5 * NP ? 2 * (u / 5) + 1 : (GS == 128 && u < 63 ? 25 : -1);
    }
    // digit of the low half (the high half holds the same digit of byte_b, or
    // digit + 1 of byte_a)
    __host__ __device__ static constexpr int digit(int u)
    {
        return u < 5 * NP ? u % 5 : (GS == 64 ? (u == 30 ? 0 : 2) : (u < 63 ? u - 60 : 3));
    }
    __host__ __device__ static constexpr int code_lo(int u) { return 5 * byte_a(u) + digit(u); }
    __host__ __device__ static constexpr int code_hi(int u)
    {
        return byte_b(u) >= 0 ? 5 * byte_b(u) + digit(u) : 5 * byte_a(u) + digit(u) + 1;
    }
};

// every code of a group is exactly one half of one item
template <int GS>
constexpr bool items_cover_group()
{
    bool seen[GS] = {};
    for (int u = 0; u < GS / 2; ++u) {
        const int lo = T5G<GS>::code_lo(u), hi = T5G<GS>::code_hi(u);
        if (lo < 0 || lo >= GS || hi < 0 || hi >= GS || lo == hi || seen[lo] || seen[hi]) return false;
        seen[lo] = seen[hi] = true;
    }
    return true;
}
static_assert(items_cover_group<64>() && items_cover_group<128>(), "t5 item plan must cover every code once");
static_assert(T5G<64>::NG * T5G<64>::MPG == kMmasR && T5G<128>::NG * T5G<128>::MPG == kMmasR,
              "a chunk is kMmasR MMAs per 16 rows");

// codes (within the group) of each item half, for the B gather table
struct T5Items {
    uint8_t lo[2][64], hi[2][64];  // [gs == 128][item]
};

constexpr T5Items make_t5_items()
{
    T5Items tb{};
    for (int u = 0; u < 32; ++u) {
        tb.lo[0][u] = (uint8_t)T5G<64>::code_lo(u);
        tb.hi[0][u] = (uint8_t)T5G<64>::code_hi(u);
    }
    for (int u = 0; u < 64; ++u) {
        tb.lo[1][u] = (uint8_t)T5G<128>::code_lo(u);
        tb.hi[1][u] = (uint8_t)T5G<128>::code_hi(u);
    }
    return tb;
}

__constant__ T5Items c_t5 = make_t5_items();

// stage layout: weights [rows][208] | scales [rows][GPC] | biases (if any)
// | B fragments [32][M][4] uint4 | then either the group sums (hi, lo)
// [NB][M][4] uint2 of the bias MMAs, or (column split) {Sx, Cx} of x rows
// 0, 1 per (period, slot) [NG][4] float4 and 64 zero bytes (128-aligned)
template <int GS, bool HAS_BIAS, bool COL, int NW>
struct Stage5 {
    static constexpr int kW = Cta<NW>::kRows * kBytesR;
    static constexpr int kS = Cta<NW>::kRows * T5G<GS>::GPC * 2;
    static constexpr int kScale = kW;
    static constexpr int kBias = kW + kS;
    static constexpr int kB = kW + kS * (HAS_BIAS ? 2 : 1);
    __host__ __device__ static constexpr int sx_off(int M) { return kB + kPairsR * M * 64; }
    __host__ __device__ static constexpr int zero_off(int M) { return (sx_off(M) + T5G<GS>::NG * 4 * 16 + 127) / 128 * 128; }
    __host__ __device__ static constexpr int bytes(int M)
    {
        return ((COL ? zero_off(M) + 64 : sx_off(M) + T5G<GS>::NB * M * 32) + 127) / 128 * 128;
    }
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

// 16 bytes global -> shared through the load/store path (src_bytes 0: zeros);
// a thread's copies complete at its cp.async.wait_all
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void sts128(uint32_t a, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// loads of data written before the stage's full barrier completed (ordered by
// the volatile wait that precedes them in program order)
__device__ __forceinline__ uint4 lds128r(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t lds32r(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint2 lds64r(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ void mma_r(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a0, a1) = fma(s, (d0 + e0, d1 + e1) - (c0, c1), fma(b, (x0, x1), (a0, a1)))
// on packed fp32 pairs: each element rounds as the scalar operations would
__device__ __forceinline__ void col_epi2(float &a0, float &a1, float s, float b, float d0, float d1, float e0, float e1,
                                         float c0, float c1, float x0, float x1)
{
    asm("{\n\t.reg .b64 d, e, c, x, a, ss, bb;\n\t"
        "mov.b64 d, {%2, %3};\n\t"
        "mov.b64 e, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\t"
        "mov.b64 x, {%8, %9};\n\t"
        "mov.b64 ss, {%10, %10};\n\t"
        "mov.b64 bb, {%11, %11};\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "add.rn.f32x2 d, d, e;\n\t"
        "sub.rn.f32x2 d, d, c;\n\t"
        "fma.rn.f32x2 a, bb, x, a;\n\t"
        "fma.rn.f32x2 a, ss, d, a;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(d0), "f"(d1), "f"(e0), "f"(e1), "f"(c0), "f"(c1), "f"(x0), "f"(x1), "f"(s), "f"(b));
}

// one or two floats into CTA `rank`'s shared memory; each write completes
// its bytes on that CTA's mbarrier at the same local offset as `local_bar`
__device__ __forceinline__ void st_async_f32r(uint32_t local_addr, uint32_t local_bar, uint32_t rank, float a)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(ra), "f"(a), "r"(rb)
                 : "memory");
}

__device__ __forceinline__ void st_async_v2r(uint32_t local_addr, uint32_t local_bar, uint32_t rank, float a, float b)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(ra),
                 "f"(a), "f"(b), "r"(rb)
                 : "memory");
}

// fp16x2 constants of the decode (in registers)
struct T5Consts {
    uint32_t third;  // (1/3, 1/3)
    uint32_t c682;   // (682.5, 682.5)
    uint32_t m3;     // (-3, -3)
    uint32_t e64;    // 0x64006400: the exponent byte of 1024 in both halves
};

// 1024 + byte as fp16 of slice bytes oa (low half) and ob (high half)
__device__ __forceinline__ uint32_t v_pair(const uint32_t (&w)[13], int oa, int ob, uint32_t e64)
{
    const int wa = oa >> 2, wb = ob >> 2;
    if (wa == wb) return __byte_perm(w[wa], e64, (uint32_t)((oa & 3) | (5 << 4) | ((ob & 3) << 8) | (7 << 12)));
    const uint32_t v = __byte_perm(w[wa], w[wb], (uint32_t)((oa & 3) | ((4 + (ob & 3)) << 8)));
    return __byte_perm(v, e64, 0x7250u);
}

// The A register of item u of group period P for one row whose slice words are
// w[13] (bytes 52t .. 52t+51 of the row's chunk), before scaling: t - 2048 in
// each half, or t + 1024 for digit 4 of a pair.  Called in fully unrolled
// loops: P and u fold to constants (w[] stays in registers, selectors are
// immediates) and the divisions shared by a pair's five items merge.
template <int GS>
__device__ __forceinline__ uint32_t item_raw(int P, int u, const uint32_t (&w)[13], const T5Consts &k)
{
    using Ge = T5G<GS>;
    const int oa = Ge::B * P + Ge::byte_a(u);
    const int d = Ge::digit(u);
    uint32_t q[6];
    if (Ge::byte_b(u) >= 0) {
        q[0] = v_pair(w, oa, Ge::B * P + Ge::byte_b(u), k.e64);
    } else {
        // digits d, d+1 of one byte: the high half starts one division ahead
        // (gs=128: byte 24 is also the low byte of the pair (24, 25))
        const uint32_t v = v_pair(w, oa, GS == 128 ? Ge::B * P + 25 : oa, k.e64);
        q[0] = __byte_perm(v, hfma2(v, k.third, k.c682), 0x5410);
    }
#pragma unroll
    for (int j = 0; j < 5; ++j)
        if (j <= d) q[j + 1] = hfma2(q[j], k.third, k.c682);
    return d < 4 || Ge::byte_b(u) < 0 ? hfma2(q[d + 1], k.m3, q[d]) : q[4];
}

// offset class of item u: 0 = t - 2048, 1 = t + 1024
template <int GS>
__host__ __device__ constexpr int item_off(int u)
{
    return T5G<GS>::byte_b(u) >= 0 && T5G<GS>::digit(u) == 4 ? 1 : 0;
}

// fp16(s t) from an item: fma(A, s, -off s) is exact while |s| < 32; else (A - off) s
template <bool FAST>
__device__ __forceinline__ uint32_t scale_item(uint32_t a, uint32_t s2, uint32_t ks2, uint32_t off2)
{
    return FAST ? hfma2(a, s2, ks2) : hmul2(hsub2(a, off2), s2);
}

// COL: column split (passes of M <= 2 x rows), see the file comment
template <int GS, bool HAS_BIAS, bool COL, int NW>
__global__ void __launch_bounds__(Cta<NW>::kThreads, Cta<NW>::kPerSM)
    qmv_t5r_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap bmap, const T5RParams p)
{
    using Ge = T5G<GS>;
    using SL = Stage5<GS, HAS_BIAS, COL, NW>;
    constexpr int kRowsR = Cta<NW>::kRows;
    constexpr int kThreadsR = Cta<NW>::kThreads;
    constexpr int NG = Ge::NG;
    constexpr int GPC = Ge::GPC;
    constexpr int MPG = Ge::MPG;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStagesR], empty_bar[kMaxStagesR];
    __shared__ __align__(8) uint64_t red_bar;  // split K: this rank's rows of every rank's partials have landed
    __shared__ __align__(16) uint16_t koff[kPairsR * 4 * 8];  // (pair, slot, half) -> staging offset
    __shared__ int last_it[kMaxStagesR];  // iteration whose weights a stage received last (-1: none)

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

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_a = smem_addr(smem);
    const uint32_t xraw_a = ring_a + (uint32_t)NST * STB;  // 2 x [M][1024] fp16: producer pw's buffer is pw
    const uint32_t XB = (uint32_t)(M * kCodesR * 2);
    float *red = reinterpret_cast<float *>(smem + (size_t)NST * STB + 2 * (size_t)XB);  // [S][RS][8]

    // B fragment column of this thread.  Plain: x row g (columns >= M read a
    // valid row; their outputs are dropped).  Column split: column g is x
    // row g & 1 at the k-slots of thread g >> 1, so this thread's entries
    // exist only when g >> 1 == t; otherwise it reads the stage's zero bytes.
    const int mcol = min(g, M - 1);
    uint32_t bqo = (uint32_t)(SL::kB + (mcol * 4 + t) * 16);
    uint32_t bstride = (uint32_t)(M * 64);
    if constexpr (COL) {
        // (the zero granule of lane pair g >> 1 avoids the banks that the active
        // thread of its quarter-warp reads: no conflict between the two)
        const bool act = (g >> 1) == t && (g & 1) < M;
        bqo = act ? (uint32_t)(SL::kB + ((g & 1) * 4 + t) * 16) : (uint32_t)(SL::zero_off(M) + (((g >> 1) + 2) & 3) * 16);
        bstride = act ? (uint32_t)(M * 64) : 0u;
    }

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 33);  // producer lane 0 (expect_tx) + 32 once x is prepared
            mbar_init(smem_addr(&empty_bar[s]), NW * 32);
        }
        if (S > 1) {
            // rows [rank RS, rank RS + nrow) from all S ranks: M floats a row
            // (column split), else ceil(M/2) float pairs
            const int nrow = max(0, min(p.RS, kRowsR - rank * p.RS));
            const int row_bytes = COL ? 4 * M : 8 * ((M + 1) / 2);
            mbar_init(smem_addr(&red_bar), 1);
            mbar_arrive_expect_tx(smem_addr(&red_bar), (uint32_t)(S * nrow * row_bytes));
        }
    }
    if constexpr (COL) {
        for (int i = tid; i < 4 * NST; i += kThreadsR)
            sts128(ring_a + (uint32_t)(i >> 2) * STB + (uint32_t)(SL::zero_off(M) + (i & 3) * 16), make_uint4(0, 0, 0, 0));
    }
    // B gather table: entry (pair ip, slot, q) is half q & 1 of item 2i + ((q >> 1) & 1)
    // of MMA 2ip + (q >> 2) = period pp, MMA i; staging layout [box k/256][x row][256]
    for (int e = tid; e < kPairsR * 4 * 8; e += kThreadsR) {
        const int q = e & 7, slot = (e >> 3) & 3, ip = e >> 5;
        const int i0 = 2 * ip + (q >> 2);
        const int pp = i0 / MPG, i = i0 % MPG;
        const int u = 2 * i + ((q >> 1) & 1);
        const int code = (q & 1) ? c_t5.hi[GS == 128][u] : c_t5.lo[GS == 128][u];
        const int kc = (NG * slot + pp) * GS + code;
        koff[e] = (uint16_t)((kc >> 8) * M * 512 + (kc & 255) * 2);
    }
    if (tid < kMaxStagesR) last_it[tid] = -1;
    __syncthreads();
    // split phase: every CTA of the cluster has started, with its reduction
    // barrier set up, before any distributed-shared-memory store (the matching
    // wait is before them)
    if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    if (warp >= NW) {
        // ---- producers: pw prepares chunks pw, pw + 2, ... from x buffer pw -----------
        const int pw = warp - NW;
        auto issue = [&](int it, int s) {
            if (lane == 0) {
                last_it[s] = it;
                const uint32_t bar = smem_addr(&full_bar[s]);
                const uint32_t st = ring_a + (uint32_t)s * STB;
                mbar_arrive_expect_tx(bar, (uint32_t)(SL::kW + SL::kS * (HAS_BIAS ? 2 : 1)));
                const int c = c_lo + it;
                tma_2d(st, &wmap, c * kBytesR, n0, bar);
                tma_2d(st + SL::kScale, &smap, c * GPC, n0, bar);
                if (HAS_BIAS) tma_2d(st + SL::kBias, &bmap, c * GPC, n0, bar);
            }
        };
        // x of chunk `it` into staging buffer it & 1 (= pw), laid out [256-code box
        // j][x row m][256], by 16-byte copies of the warp's lanes through the
        // load/store path (a TMA copy would queue behind the weight copies);
        // a pass's rows past the call's M read as zeros
        auto issue_x = [&](int it) {
            const uint32_t xb = xraw_a + (uint32_t)(it & 1) * XB;
            const int k0 = (c_lo + it) * kCodesR + 8 * lane;
            for (int m = 0; m < M; ++m) {
                const int row = M * (int)blockIdx.y + m;
                const bool in = row < p.Mtot;
                const __half *src = p.x + (size_t)(in ? row : 0) * p.K + k0;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cp_async16(xb + (uint32_t)((j * M + m) * 512 + 16 * lane), src + 256 * j, in ? 16u : 0u);
            }
            cp_async_commit();
        };
        const int pre = min(NST, ncl);
        int issued_end = pw;  // this producer's iterations below issued_end have their weights requested
        for (int it = pw; it < pre; it += kProdR) {
            issue(it, it);
            issued_end = it + kProdR;
        }
        // indicator A rows of the group sums: row r is 1 on the k-slots of
        // group r (thread t's slots of period P hold group NG t + P)
        uint32_t ind0[NG], ind1[NG];
#pragma unroll
        for (int P = 0; P < NG; ++P) {
            ind0[P] = g == NG * t + P ? 0x3C003C00u : 0u;
            ind1[P] = g + 8 == NG * t + P ? 0x3C003C00u : 0u;
        }
        // column split: A row 0 ones, row 1 the item offset (-2048, or +1024 for
        // digit 4 of a pair) in both halves, rows 2..15 zero
        uint32_t aofs[2];
        aofs[0] = g == 0 ? 0x3C003C00u : (g == 1 ? (0xE800E800u ^ p.zero) : 0u);
        aofs[1] = g == 0 ? 0x3C003C00u : (g == 1 ? (0x64006400u ^ p.zero) : 0u);
        __syncwarp();
        pdl_wait();
        if (pw < ncl) issue_x(pw);
        int done = pw;  // this producer's iterations below done are prepared
        for (int it = pw; it < ncl; it += kProdR) {
            const int s = it % NST;
            const uint32_t par = (uint32_t)(it / NST) & 1u;
            const uint32_t st = ring_a + (uint32_t)s * STB;
            if (it >= NST) {
                bool ok = lane == 0 ? wait_bounded_r(smem_addr(&empty_bar[s]), par ^ 1u, p.wait_ns) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                issue(it, s);
                issued_end = it + kProdR;
            }
            // x of chunk it: each lane's copies, then every lane's
            cp_async_wait_all();
            __syncwarp();
            const uint32_t xb = xraw_a + (uint32_t)(it & 1) * XB;
            // B fragments: entry (ip, x row m, slot) at kB + ((ip M + m) 4 + slot) 16.
            // Each pass of the warp gathers from one x row (rows are 512 bytes
            // apart in the staging buffer: mixing them would stack bank conflicts)
            // (two passes at a time: their 16 gathers are issued before either
            // store, so that their latencies overlap)
            for (int k = 0; k < 4 * M; k += 2) {
                uint32_t h[2][8];
                int e[2];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int m = (k + kk) >> 2, el = (((k + kk) & 3) << 5) | lane;
                    const int ip = el >> 2, slot = el & 3;
                    e[kk] = (ip * M + m) * 4 + slot;
                    const uint4 kw = *reinterpret_cast<const uint4 *>(&koff[(ip * 4 + slot) * 8]);
                    const uint32_t xm = xb + (uint32_t)(512 * m);
                    const uint32_t o[8] = {xm + (kw.x & 0xffffu), xm + (kw.x >> 16), xm + (kw.y & 0xffffu),
                                           xm + (kw.y >> 16),     xm + (kw.z & 0xffffu), xm + (kw.z >> 16),
                                           xm + (kw.w & 0xffffu), xm + (kw.w >> 16)};
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint16_t v16;
                        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v16) : "r"(o[q]));
                        h[kk][q] = v16;
                    }
                }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    sts128(st + SL::kB + (uint32_t)(e[kk] * 16),
                           make_uint4(__byte_perm(h[kk][0], h[kk][1], 0x5410), __byte_perm(h[kk][2], h[kk][3], 0x5410),
                                      __byte_perm(h[kk][4], h[kk][5], 0x5410), __byte_perm(h[kk][6], h[kk][7], 0x5410)));
            }
            // every lane's reads of the buffer are done before any lane's copy
            // of this producer's next chunk rewrites it
            __syncwarp();
            if (it + kProdR < ncl) issue_x(it + kProdR);
            if constexpr (COL) {
                // Sx (row 0) and Cx (row 1) of every (period, slot, x row): the
                // consumers' MMA sequence (two chains per period) over a constant A.
                // The periods' chains are interleaved (each keeps its own order, so
                // the sums are the consumers' bit for bit): one warp runs them, and
                // period after period their latencies would add up
                float d2[NG][2][4];
#pragma unroll
                for (int P = 0; P < NG; ++P)
#pragma unroll
                    for (int q = 0; q < 4; ++q) d2[P][0][q] = d2[P][1][q] = 0.f;
#pragma unroll
                for (int i = 0; i < MPG; i += 2) {
#pragma unroll
                    for (int P = 0; P < NG; ++P) {
                        const int ic = P * MPG + i;
                        const uint4 bv = lds128r(st + bqo + (uint32_t)(ic >> 1) * bstride);
                        mma_r(d2[P][(i >> 1) & 1], aofs[item_off<GS>(2 * i)], 0u, aofs[item_off<GS>(2 * i + 1)], 0u, bv.x,
                              bv.y);
                        mma_r(d2[P][(i >> 1) & 1], aofs[item_off<GS>(2 * i + 2)], 0u, aofs[item_off<GS>(2 * i + 3)], 0u,
                              bv.z, bv.w);
                    }
                }
                if (g < 2) {
#pragma unroll
                    for (int P = 0; P < NG; ++P) {
                        const uint32_t a = st + (uint32_t)SL::sx_off(M) + (uint32_t)((P * 4 + t) * 16 + 4 * g);
                        // float4 {Sx(x row 0), Cx(0), Sx(1), Cx(1)}: thread g writes elements g, g + 2
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(d2[P][0][0] + d2[P][1][0]) : "memory");
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(a + 8), "f"(d2[P][0][1] + d2[P][1][1]) : "memory");
                    }
                }
            } else {
                // group sums on the tensor core: D[r][m] = Sx[group r][x row m];
                // thread (g, t) holds groups g, g+8 of x rows 2t, 2t+1
                {
                    // eight accumulator chains, one warp: their latencies overlap
                    float d4[8][4];
#pragma unroll
                    for (int q = 0; q < 8; ++q) d4[q][0] = d4[q][1] = d4[q][2] = d4[q][3] = 0.f;
#pragma unroll
                    for (int P = 0; P < NG; ++P)
#pragma unroll
                        for (int i = 0; i < MPG; i += 2) {
                            const int ic = P * MPG + i;
                            const uint4 bv = lds128r(st + bqo + (uint32_t)(ic >> 1) * bstride);
                            mma_r(d4[(ic >> 1) & 7], ind0[P], ind1[P], ind0[P], ind1[P], bv.x, bv.y);
                            mma_r(d4[(ic >> 1) & 7], ind0[P], ind1[P], ind0[P], ind1[P], bv.z, bv.w);
                        }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = g + 8 * (q >> 1), m = 2 * t + (q & 1);
                        if (r < GPC && m < M) {
                            const float v =
                                ((d4[0][q] + d4[1][q]) + (d4[2][q] + d4[3][q])) + ((d4[4][q] + d4[5][q]) + (d4[6][q] + d4[7][q]));
                            const __half hi = __float2half_rn(v);
                            const __half lo = __float2half_rn(v - __half2float(hi));
                            // bias MMA nb: slots 2t, 2t+1 <- group NG t + 2nb, slots 2t+8, 2t+9 <- group NG t + 2nb + 1
                            const int slot = r / NG, rem = r % NG, nb = rem >> 1, h2 = rem & 1;
                            const uint32_t a = st + (uint32_t)SL::sx_off(M) + (uint32_t)(((nb * M + m) * 4 + slot) * 8 + 4 * h2);
                            asm volatile("st.shared.u32 [%0], %1;" ::"r"(a),
                                         "r"((uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16))
                                         : "memory");
                        }
                    }
                }
            }
            __syncwarp();
            mbar_arrive_r(smem_addr(&full_bar[s]));
            done = it + kProdR;
        }
        // every copy this CTA issued has landed before anyone leaves: this
        // producer's stages whose weights were requested but that were never
        // prepared (a wait expired) get their missing arrivals; once both
        // producers have stopped issuing, each awaits the stages it filled last
        // (and each lane its x copies still in flight)
        for (int it = done; it < issued_end; it += kProdR) mbar_arrive_r(smem_addr(&full_bar[it % NST]));
        asm volatile("bar.sync 1, %0;" ::"n"(kProdR * 32) : "memory");
        if (lane == 0) {
            for (int s = 0; s < NST; ++s) {
                const int li = last_it[s];
                if (li >= 0 && li % kProdR == pw)
                    wait_bounded_r(smem_addr(&full_bar[s]), (uint32_t)(li / NST) & 1u, kDrainWaitNs);
            }
        }
        cp_async_wait_all();
        __syncwarp();
        if (S > 1) {
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
        }
        return;
    }

    // ---- consumers -------------------------------------------------------------------
    T5Consts kc;
    kc.third = 0x35553555u ^ p.zero;
    kc.c682 = 0x61556155u ^ p.zero;
    kc.m3 = 0xC200C200u ^ p.zero;
    kc.e64 = 0x64006400u ^ p.zero;
    const uint32_t c2048 = 0x68006800u ^ p.zero, cm1024 = 0xE400E400u ^ p.zero;  // (2048, 2048), (-1024, -1024)
    const uint32_t off0 = 0xE800E800u ^ p.zero, off1 = 0x64006400u ^ p.zero;    // item offsets -2048, +1024
    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
    const int r0 = warp * 16 + g;
    uint32_t st_a = ring_a;
    int s = 0;
    uint32_t par = 0;
    for (int it = 0; it < ncl; ++it) {
        if (!wait_bounded_r(smem_addr(&full_bar[s]), par, p.wait_ns)) break;
        // scales (and biases) of this thread's groups NG t .. NG t + NG - 1, rows r0, r0+8
        uint32_t sw[2][NG / 2], bw[2][NG / 2];
        bool fast = true;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint32_t sa = st_a + SL::kScale + (uint32_t)(((r0 + 8 * rr) * GPC + NG * t) * 2);
            if constexpr (NG == 4) {
                const uint2 v = lds64r(sa);
                sw[rr][0] = v.x;
                sw[rr][1] = v.y;
                if constexpr (HAS_BIAS) {
                    const uint2 b = lds64r(sa + SL::kS);
                    bw[rr][0] = b.x;
                    bw[rr][1] = b.y;
                }
            } else {
                sw[rr][0] = lds32r(sa);
                if constexpr (HAS_BIAS) bw[rr][0] = lds32r(sa + SL::kS);
            }
#pragma unroll
            for (int q = 0; q < NG / 2; ++q) {
                const __half2 h = *reinterpret_cast<const __half2 *>(&sw[rr][q]);
                fast = fast && fabsf(__low2float(h)) < 32.f && fabsf(__high2float(h)) < 32.f;
            }
        }
        const uint32_t bq = st_a + bqo;
        const uint32_t wra = st_a + (uint32_t)(r0 * kBytesR + kSliceR * t);
        if constexpr (COL) {
            // per period: D[n][2t+e] = x row e . (t_d - 2048 or t_4 + 1024) over this
            // thread's group NG t + P, two MMA chains; then s (D - Cx) + b Sx in fp32
            uint32_t wa[13], wb[13];
#pragma unroll
            for (int P = 0; P < NG; ++P) {
#pragma unroll
                for (int q = 0; q < 13; ++q) {
                    const bool need = q >= (Ge::B * P) / 4 && q <= (Ge::B * P + Ge::B - 1) / 4;
                    const bool had = P > 0 && q <= (Ge::B * P - 1) / 4;
                    if (need && !had) {
                        wa[q] = lds32r(wra + (uint32_t)(4 * q));
                        wb[q] = lds32r(wra + (uint32_t)(8 * kBytesR + 4 * q));
                    }
                }
                float d2[2][4];
#pragma unroll
                for (int q = 0; q < 4; ++q) d2[0][q] = d2[1][q] = 0.f;
#pragma unroll
                for (int i = 0; i < MPG; i += 2) {
                    const uint32_t a0 = item_raw<GS>(P, 2 * i, wa, kc), a1 = item_raw<GS>(P, 2 * i, wb, kc);
                    const uint32_t a2 = item_raw<GS>(P, 2 * i + 1, wa, kc), a3 = item_raw<GS>(P, 2 * i + 1, wb, kc);
                    const uint32_t c0 = item_raw<GS>(P, 2 * i + 2, wa, kc), c1 = item_raw<GS>(P, 2 * i + 2, wb, kc);
                    const uint32_t c2 = item_raw<GS>(P, 2 * i + 3, wa, kc), c3 = item_raw<GS>(P, 2 * i + 3, wb, kc);
                    const int ic = P * MPG + i;
                    const uint4 bv = lds128r(bq + (uint32_t)(ic >> 1) * bstride);
                    mma_r(d2[(i >> 1) & 1], a0, a1, a2, a3, bv.x, bv.y);
                    mma_r(d2[(i >> 1) & 1], c0, c1, c2, c3, bv.z, bv.w);
                }
                float sc[2], bi[2];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint32_t sv = sw[rr][P >> 1];
                    const __half sh = __ushort_as_half((uint16_t)((P & 1) ? (sv >> 16) : (sv & 0xffffu)));
                    sc[rr] = __half2float(sh);
                    if constexpr (HAS_BIAS) {
                        const uint32_t bv2 = bw[rr][P >> 1];
                        bi[rr] = __half2float(__ushort_as_half((uint16_t)((P & 1) ? (bv2 >> 16) : (bv2 & 0xffffu))));
                    } else {
                        bi[rr] = __half2float(sym_bias(sh, p.ratio));
                    }
                }
                const uint4 v = lds128r(st_a + (uint32_t)SL::sx_off(M) + (uint32_t)((P * 4 + t) * 16));
                const float sx[2] = {__uint_as_float(v.x), __uint_as_float(v.z)};
                const float cx[2] = {__uint_as_float(v.y), __uint_as_float(v.w)};
                // value q: row half q >> 1 (scale and bias rr), x row q & 1
                col_epi2(acc[0][0], acc[0][1], sc[0], bi[0], d2[0][0], d2[0][1], d2[1][0], d2[1][1], cx[0], cx[1], sx[0],
                         sx[1]);
                col_epi2(acc[0][2], acc[0][3], sc[1], bi[1], d2[0][2], d2[0][3], d2[1][2], d2[1][3], cx[0], cx[1], sx[0],
                         sx[1]);
            }
        } else {

            // the chunk's 64 MMAs; FAST: scaled items by one HFMA2 each
            auto body = [&](auto fast_tag) {
                constexpr bool kFast = decltype(fast_tag)::value;
                uint32_t wa[13], wb[13];
#pragma unroll
                for (int P = 0; P < NG; ++P) {
                    // words holding bytes [B P, B P + B) of the slices (the first may
                    // have been read for the previous group)
#pragma unroll
                    for (int q = 0; q < 13; ++q) {
                        const bool need = q >= (Ge::B * P) / 4 && q <= (Ge::B * P + Ge::B - 1) / 4;
                        const bool had = P > 0 && q <= (Ge::B * P - 1) / 4;
                        if (need && !had) {
                            wa[q] = lds32r(wra + (uint32_t)(4 * q));
                            wb[q] = lds32r(wra + (uint32_t)(8 * kBytesR + 4 * q));
                        }
                    }
                    // this group's scale in both halves, and -off * scale for the two offsets
                    uint32_t s2[2], k0[2], k1[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        s2[rr] = __byte_perm(sw[rr][P >> 1], 0u, (P & 1) ? 0x3232u : 0x1010u);
                        k0[rr] = hmul2(s2[rr], c2048);
                        k1[rr] = hmul2(s2[rr], cm1024);
                    }
#pragma unroll
                    for (int i = 0; i < MPG; i += 2) {
                        uint32_t A[2][4];
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int u = 2 * (i + h) + hh;
                                const bool o1 = item_off<GS>(u) == 1;
                                A[h][2 * hh] = scale_item<kFast>(item_raw<GS>(P, u, wa, kc), s2[0], o1 ? k1[0] : k0[0],
                                                                 o1 ? off1 : off0);
                                A[h][2 * hh + 1] = scale_item<kFast>(item_raw<GS>(P, u, wb, kc), s2[1], o1 ? k1[1] : k0[1],
                                                                     o1 ? off1 : off0);
                            }
                        const int ic = P * MPG + i;
                        const uint4 bv = lds128r(bq + (uint32_t)(ic >> 1) * bstride);
                        mma_r(acc[(ic >> 1) & 3], A[0][0], A[0][1], A[0][2], A[0][3], bv.x, bv.y);
                        mma_r(acc[(ic >> 1) & 3], A[1][0], A[1][1], A[1][2], A[1][3], bv.z, bv.w);
                    }
                }
            };
            if (__all_sync(0xffffffffu, fast)) body(std::true_type{});
            else body(std::false_type{});

            // bias term: slots 2t, 2t+1 <- group NG t + 2nb, slots 2t+8, 2t+9 <- group NG t + 2nb + 1
            const uint32_t sq = st_a + (uint32_t)SL::sx_off(M) + (uint32_t)((mcol * 4 + t) * 8);
#pragma unroll
            for (int nb = 0; nb < Ge::NB; ++nb) {
                uint32_t bb[2][2];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint32_t bsrc = HAS_BIAS ? bw[rr][nb] : sw[rr][nb];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint16_t v16 = (uint16_t)(bsrc >> (16 * h));
                        bb[rr][h] = HAS_BIAS ? dup_half(v16)
                                             : dup_half(__half_as_ushort(sym_bias(__ushort_as_half(v16), p.ratio)));
                    }
                }
                const uint2 bxy = lds64r(sq + (uint32_t)(nb * M * 32));
                mma_r(acc[nb & 3], bb[0][0], bb[1][0], bb[0][1], bb[1][1], bxy.x, bxy.y);
            }
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
    // column split: the four threads of a quad hold four groups of the same
    // rows and x rows; add them (fixed order), then thread t writes row
    // r0 + 8 (t >> 1), x row t & 1
    const int rr_t = t >> 1, e_t = t & 1;
    float vcol = 0.f;
    if constexpr (COL) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[q] += __shfl_xor_sync(0xffffffffu, v[q], 1);
            v[q] += __shfl_xor_sync(0xffffffffu, v[q], 2);
        }
        vcol = rr_t ? (e_t ? v[3] : v[2]) : (e_t ? v[1] : v[0]);
    }

    // ---- results: value q is row r0 + 8 (q >> 1), x row 2t + (q & 1) -------------------
    const int Mv = min(M, p.Mtot - M * (int)blockIdx.y);  // rows of this pass that exist
    __half *outg = p.out + (size_t)(M * blockIdx.y) * p.N;
    if (S == 1) {
        if constexpr (COL) {
            const int n = n0 + r0 + 8 * rr_t;
            if (n < p.N && e_t < Mv) outg[(size_t)e_t * p.N + n] = __float2half_rn(vcol);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = n0 + r0 + 8 * (q >> 1), m = 2 * t + (q & 1);
                if (n < p.N && m < Mv) outg[(size_t)m * p.N + n] = __float2half_rn(v[q]);
            }
        }
        return;
    }
    // reduce-scatter: each rank sends its values with st.async, completing
    // bytes of the receiving rank's red_bar; a rank adds its rows once all
    // have landed.  The cluster barrier split around the reduction keeps
    // every CTA resident until every rank has received all of its rows.
    const int RS = p.RS;
    const uint32_t rbar = smem_addr(&red_bar);
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if constexpr (COL) {
        const int row = r0 + 8 * rr_t;
        const int q = row / RS;
        if (e_t < M) st_async_f32r(smem_addr(red + ((size_t)rank * RS + (row - q * RS)) * 8 + e_t), rbar, (uint32_t)q, vcol);
    } else if (2 * t < M) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = r0 + 8 * h;
            const int q = row / RS;
            st_async_v2r(smem_addr(red + ((size_t)rank * RS + (row - q * RS)) * 8 + 2 * t), rbar, (uint32_t)q, v[2 * h],
                         v[2 * h + 1]);
        }
    }
    // every rank sends all of its rows whatever its own waits did, so this
    // wait keeps the long limit of the drains
    wait_bounded_r(rbar, 0, kDrainWaitNs);
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const int row0 = rank * RS;
    const int nrow = max(0, min(RS, kRowsR - row0));
    for (int i = tid; i < nrow * M; i += NW * 32) {
        const int lr = i / M, m = i % M;
        float sum = 0.f;
        for (int k = 0; k < S; ++k) sum += red[((size_t)k * RS + lr) * 8 + m];
        const int n = n0 + row0 + lr;
        if (n < p.N && m < Mv) outg[(size_t)m * p.N + n] = __float2half_rn(sum);
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
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
               int64_t row_bytes, int box_cols, int box_rows)
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

template <int GS, bool HAS_BIAS, bool COL, int NW>
size_t t5r_smem(int M, int S, int stages, int RS)
{
    return 1024 + (size_t)stages * Stage5<GS, HAS_BIAS, COL, NW>::bytes(M) + 2 * (size_t)M * kCodesR * 2 + (size_t)S * RS * 8 * 4;
}

template <int GS, bool HAS_BIAS, bool COL, int NW>
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
    auto kern = qmv_t5r_kernel<GS, HAS_BIAS, COL, NW>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cta<NW>::kSmemBudget);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(Cta<NW>::kThreads);
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
template <int GS, bool HAS_BIAS, bool COL, int NW>
bool plan_r(int M, int N, int chunks, int P, RPlan &best)
{
    constexpr int kRowsR = Cta<NW>::kRows;
    constexpr size_t kSmemBudgetR = Cta<NW>::kSmemBudget;
    const int R = (N + kRowsR - 1) / kRowsR;
    const int sms = sm_count();
    const size_t stage = Stage5<GS, HAS_BIAS, COL, NW>::bytes(M);
    double best_cost = 1e30;
    bool found = false;
    for (int S = 1; S <= kMaxSplitR && S <= chunks; ++S) {
        const int Cs = (chunks + S - 1) / S;
        if ((S - 1) * Cs >= chunks) continue;
        const int RS = (kRowsR + S - 1) / S;
        // every rank owns rows of the reduction (128 rows over 14 ranks would
        // leave the last one none)
        if ((S - 1) * RS >= kRowsR) continue;
        const size_t fixed = t5r_smem<GS, HAS_BIAS, COL, NW>(M, S, 0, RS);
        if (fixed + stage > kSmemBudgetR) continue;
        int st = (int)((kSmemBudgetR - fixed) / stage);
        st = std::min(st, kMaxStagesR);
        st = std::min(st, Cs);
        if (st < 1) continue;
        const size_t sm = t5r_smem<GS, HAS_BIAS, COL, NW>(M, S, st, RS);
        const int slots = S == 1 ? Cta<NW>::kPerSM * sms : cluster_slots_r<GS, HAS_BIAS, COL, NW>(S, sm);
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

template <int GS, bool HAS_BIAS, bool COL, int NW>
int launch_r(const T5RParams &p0, int64_t row_bytes, cudaStream_t s)
{
    CUtensorMap wmap;
    if (!encode_2d(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, p0.w, row_bytes, p0.N, row_bytes, kBytesR, Cta<NW>::kRows))
        return BQD_ERR_UNSUPPORTED;
    RPlan pl;
    const int P = (p0.Mtot + p0.M - 1) / p0.M;
    if (!plan_r<GS, HAS_BIAS, COL, NW>(p0.M, p0.N, p0.chunks, P, pl)) return BQD_ERR_UNSUPPORTED;
    T5RParams p = p0;
    p.S = pl.S;
    p.Cs = pl.Cs;
    p.stages = pl.stages;
    p.RS = pl.RS;
    p.stage_bytes = (uint32_t)Stage5<GS, HAS_BIAS, COL, NW>::bytes(p.M);
    constexpr int GPC = T5G<GS>::GPC;
    CUtensorMap smap, bmap;
    if (!encode_2d(smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.scales, p.G, p.N, (int64_t)p.G * 2, GPC, Cta<NW>::kRows))
        return BQD_ERR_CUDA;
    bmap = smap;
    if (HAS_BIAS && !encode_2d(bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.biases, p.G, p.N, (int64_t)p.G * 2, GPC, Cta<NW>::kRows))
        return BQD_ERR_CUDA;
    if (opt_debug_plan())
        fprintf(stderr, "bqd t5r plan: N=%d K=%d M=%d (%d per pass) gs=%d col=%d rows=%d -> S=%d Cs=%d stages=%d R=%d grid=%dx%d smem=%zu\n",
                p.N, p.K, p.Mtot, p.M, GS, (int)COL, Cta<NW>::kRows, pl.S, pl.Cs, pl.stages, pl.R, pl.R * pl.S, P, pl.smem);
    auto kern = qmv_t5r_kernel<GS, HAS_BIAS, COL, NW>;
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cta<NW>::kSmemBudget) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.R * pl.S, P);
    cfg.blockDim = dim3(Cta<NW>::kThreads);
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
    return cudaLaunchKernelEx(&cfg, kern, wmap, smap, bmap, p) == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
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
    T5RParams p;
    p.w = static_cast<const uint8_t *>(a.w);
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
    // passes of at most two x rows take the column split (no per-weight
    // scaling).  Passes of up to five rows run 128-row CTAs, two per SM: a CTA
    // that finishes frees room for the next kernel's first weight copies
    // (programmatic dependent launch), which a 256-row CTA holding most of the
    // SM's shared memory would block.  Passes of six or more rows need the
    // larger B-fragment and x buffers of one 256-row CTA per SM.
    const bool col = p.M <= 2;
    const bool narrow = p.M <= 5;
    const int64_t rb = a.row_bytes;
#define BQD_T5R_LAUNCH(GSV, HBV)                                                                                 \
    (col ? (narrow ? launch_r<GSV, HBV, true, 8>(p, rb, s) : launch_r<GSV, HBV, true, 16>(p, rb, s))           \
         : (narrow ? launch_r<GSV, HBV, false, 8>(p, rb, s) : launch_r<GSV, HBV, false, 16>(p, rb, s)))
    int rc;
    if (a.gs == 64) rc = hb ? BQD_T5R_LAUNCH(64, true) : BQD_T5R_LAUNCH(64, false);
    else rc = hb ? BQD_T5R_LAUNCH(128, true) : BQD_T5R_LAUNCH(128, false);
#undef BQD_T5R_LAUNCH
    return rc;
}

}  // namespace bqd
