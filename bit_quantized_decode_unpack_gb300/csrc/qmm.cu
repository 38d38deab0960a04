// Prefill matrix product of packed weights on the 5th-generation tensor cores
// (tcgen05), for the t5 ternary format and the 1/2-bit affine formats.
//
// Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析", §二.3: for long
// prefill (M > 16) t5 weights go through a fused "unpack + matrix multiply"
// kernel (bonsai_t5_qmm) that reads every t5 byte once.  §二.1 notes that the
// 1-bit prefill path had no such kernel (it dequantised to float16 and called
// a dense matmul); here the 1/2-bit formats take the same fused product.
//
//   Y[m, n] = sum_k X[m, k] * W[n, k],  W[n, k] = fp16(fp16(s[n,g] * q[n,k]) + b[n,g])
//   (sym: b = fp16(-ratio * s); t5 with the default ratio 1 gives W = s*(t-1))
//
// One CTA owns 128 weight rows x BX activation rows (BX = 32, 64, 128 or 256;
// on wide layers with M > 256 two blocks of 256, K steps of 64 codes) and a
// range of K groups.  When the (weight, activation) tiles are too few to fill
// the GPU, the K range is split over the CTAs of a cluster: each rank owns a
// slice of the 32-column blocks, receives the other ranks' partials of it
// through distributed shared memory and adds them in rank order (no global
// scratch).
//
// Roles (320 threads):
//   warps 0-7  decode: thread (r, h) = (tid % 128, warp / 4) decodes half h of
//              weight row n0+r's codes per K step (a group of gs codes, or
//              half of a 128-code group in the two-block mode), forms the fp16
//              weights and stores them into the stage's A tile in the tcgen05
//              K-major 128-byte-swizzled layout.
//              t5: a half starts inside a byte (byte 0, 6, 12 or 18 of a group;
//              byte pairs decode as a unit and the half's codes are picked out
//              of them): the bytes go through a shared byte->trits table, then
//              a magic-exponent LOP3 + HFMA2 give s*t exactly, then + b.
//              1/2-bit: the half group is one aligned 4-, 8- or 16-byte load;
//              a byte is duplicated into both 16-bit halves of a word, and one
//              LOP3 per code pair places code 2i in the low half and code 2i+1
//              in the high half at different mantissa positions (offsets
//              2^(10-p) per half), so HFMA2 against per-half constants gives
//              (s*q_2i, s*q_2i+1) in natural K order, then + b.
//              After the K loop warp w drains TMEM lanes 32(w%4)..+31,
//              columns of half w/4, and stores Y.
//   warp 8     allocates TMEM; lane 0 issues tcgen05.mma (kind::f16, M=128,
//              N=BX, K=16, fp32 accumulation in TMEM) and tcgen05.commit, which
//              frees a stage once its MMAs have completed.
//   warp 9     lane 0 loads X tiles with TMA (cp.async.bulk.tensor, 128-byte
//              swizzle, zero fill past M).
// Every mbarrier wait is bounded; on expiry the CTA stops issuing work, drains
// what it issued (bounded), passes its remaining barriers and frees TMEM; the
// expiry is counted for bqd_device_status.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "bqd_internal.cuh"
#include "qmv_common.cuh"

namespace bqd {
namespace {

using namespace qmvdev;

constexpr int kDecodeWarpsQ = 8;                       // decode + epilogue warps
constexpr int kDecodeThreadsQ = kDecodeWarpsQ * 32;
constexpr int kMmaWarpQ = kDecodeWarpsQ;                // TMEM owner, MMA issuer
constexpr int kTmaWarpQ = kDecodeWarpsQ + 1;            // x tiles by TMA
constexpr int kThreadsQ = (kDecodeWarpsQ + 2) * 32;
constexpr int kMaxStagesQ = 8;
constexpr size_t kQmmSmemMax = 208 * 1024;  // dynamic; the replicated decode table is static
constexpr int kLutCopiesQ = 16;              // lane l reads copy l % 16: fewer bank conflicts

__device__ unsigned int g_qmm_timeouts = 0;

// pipeline waits give up after the call's limit; drain waits after a second
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    return mbar_wait_for(bar, parity, limit_ns, &g_qmm_timeouts);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ---- tcgen05 wrappers ------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t local_addr, uint32_t rank, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand with 128-byte swizzle:
// start address >> 4, leading byte offset (unused for swizzled K-major, 1),
// stride byte offset 1024 >> 4 (8-row groups of 128-byte rows), descriptor
// version 1 (bit 46), layout type SWIZZLE_128B (2, bits 61-63).  Stepping
// K by 16 fp16 elements moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B f16 (0),
// both K-major (bits 15, 16 = 0), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct QmmParams {
    const uint8_t *w;
    const __half *scales;
    const __half *biases;
    __half *out;
    float ratio;
    int M, N, K, G;
    long long row_bytes;
    int bx, S, gpr, stages;  // gpr: K groups per cluster rank
    uint32_t zero;           // always 0: keeps the magic constants in registers
    unsigned long long wait_ns;  // limit of the pipeline waits
};

// byte offset of 16-byte chunk c of row r inside one 128-row x 64-code
// sub-tile (128-byte rows, 8-row groups of 1024 bytes, chunk index ^ row%8)
__device__ __forceinline__ uint32_t sw128_offset(int r, int c)
{
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// NH = 2: the CTA owns two 256-column blocks of x (two N=256 accumulators,
// all 512 TMEM columns), so each decoded weight tile serves 512 columns; its
// K step is then 64 codes (half a 128-group), which keeps two stages of
// [A 16 KB | X 64 KB] in shared memory.  A 128-code t5 group is then decoded
// in quarters of 32 codes that start inside bytes 0, 6, 12 and 18 of its 26
// (codes 0, 32, 64 and 96 are digits 0, 2, 4 and 1 of those bytes).
template <int FMT, int GS, int NH>
__device__ __forceinline__ void qmm_body(const CUtensorMap &xmap, const QmmParams &p)
{
    constexpr bool T5F = FMT == BQD_FMT_T5;
    static_assert(NH == 1 || NH == 2, "one or two column blocks");
    constexpr int KS = NH == 2 ? 64 : GS;  // codes per K step
    constexpr int SPG = GS / KS;           // K steps per group (1 or 2)
    constexpr int B = GS == 64 ? 13 : 26;  // t5 bytes per group
    constexpr int NSUB = KS / 64;          // 64-code sub-tiles per K step
    constexpr int A_BYTES = 128 * KS * 2;  // A tile per stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t x_full[kMaxStagesQ], a_full[kMaxStagesQ], empty_bar[kMaxStagesQ], done_bar;
    __shared__ uint32_t tmem_base;
    // t5 byte -> trits table, entry v of copy c at v * 16 + c (1/2-bit: unused)
    __shared__ uint32_t lut[T5F ? 256 * kLutCopiesQ : 1];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.S;
    const int rank = S > 1 ? (int)cluster_ctarank() : 0;
    const int tile = blockIdx.x / S;
    const int n_tiles = (p.N + 127) / 128;
    const int nt = tile % n_tiles, mt = tile / n_tiles;
    const int C = NH * p.bx;  // x columns of the CTA
    const int n0 = nt * 128, m0 = mt * C;
    const int g_lo = rank * p.gpr;
    const int g_hi = min(p.G, g_lo + p.gpr);
    const int steps = max(0, g_hi - g_lo) * SPG;
    const int NST = p.stages;
    const uint32_t X_BYTES = (uint32_t)C * KS * 2;

    // 1024-byte aligned stage ring: [A tile | X tile] per stage
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t stage_bytes = A_BYTES + X_BYTES;

    if constexpr (T5F) {
        for (int q = tid; q < 256 * kLutCopiesQ; q += kThreadsQ) {
            int v = q / kLutCopiesQ, e = 0;
            if (v < 243)
                for (int d = 0; d < 5; ++d) {
                    e |= (v % 3) << (2 * d);
                    v /= 3;
                }
            lut[q] = (uint32_t)e;
        }
    }
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_addr(&x_full[s]), 1);
            mbar_init(smem_addr(&a_full[s]), kDecodeThreadsQ);
            mbar_init(smem_addr(&empty_bar[s]), 1);
        }
        mbar_init(smem_addr(&done_bar), 1);
        abort_flag = 0;
    }
    if (warp == kMmaWarpQ) tmem_alloc(smem_addr(&tmem_base), (uint32_t)C);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    pdl_wait();

    if (warp == kTmaWarpQ) {
        // ---- X producer ---------------------------------------------------------
        if (lane == 0) {
            int issued = 0, s = 0;
            uint32_t rpar = 1;  // parity of empty_bar[s] that frees it for step it (>= NST)
            for (int it = 0; it < steps; ++it) {
                if (it >= NST && !wait_bounded(smem_addr(&empty_bar[s]), rpar, p.wait_ns)) {
                    abort_flag = 1;
                    break;
                }
                const uint32_t bar = smem_addr(&x_full[s]);
                mbar_arrive_expect_tx(bar, X_BYTES);
                const int k = g_lo * GS + it * KS;
                uint8_t *xt = smem + (size_t)s * stage_bytes + A_BYTES;
                // column block hh, sub-tile sub: [bx rows][64 codes] at (hh NSUB + sub) bx 128 bytes
                for (int hh = 0; hh < NH; ++hh)
                    for (int sub = 0; sub < NSUB; ++sub)
                        tma_load_2d(smem_addr(xt + (hh * NSUB + sub) * p.bx * 128), &xmap, k + 64 * sub,
                                    m0 + hh * p.bx, bar);
                issued = it + 1;
                if (++s == NST) {
                    s = 0;
                    rpar ^= 1u;
                }
            }
            // every copy this CTA issued lands before anyone leaves, whether or
            // not the MMA issuer consumed it (it stops early once a wait of its
            // expires, possibly after this loop has ended).  Each slot's last
            // phase is the one waited for, so the parity is unambiguous.
            for (int it = max(0, issued - NST); it < issued; ++it)
                wait_bounded(smem_addr(&x_full[it % NST]), (it / NST) & 1, kDrainWaitNs);
        }
    } else if (warp == kMmaWarpQ) {
        // ---- MMA issuer -----------------------------------------------------------
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, p.bx);
            bool ok = true;
            int s = 0;
            uint32_t par = 0;
            for (int it = 0; it < steps; ++it) {
                ok = wait_bounded(smem_addr(&x_full[s]), par, p.wait_ns) && wait_bounded(smem_addr(&a_full[s]), par, p.wait_ns);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_addr(smem + (size_t)s * stage_bytes);
                const uint32_t x0 = a0 + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < KS / 16; ++kk) {
                    const int sub = kk >> 2, within = kk & 3;
                    const uint64_t ad = sw128_desc(a0 + sub * 16384 + within * 32);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        const uint64_t bd = sw128_desc(x0 + (hh * NSUB + sub) * p.bx * 128 + within * 32);
                        tc_mma(tmem + (uint32_t)(hh * p.bx), ad, bd, idesc, (it > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                tc_commit(smem_addr(&empty_bar[s]));
                if (++s == NST) {
                    s = 0;
                    par ^= 1u;
                }
            }
            if (!ok) abort_flag = 1;
            tc_commit(smem_addr(&done_bar));  // arrives once every issued MMA has completed
        }
    } else {
        // ---- decode warps: weight row n0 + (tid & 127); warps 0-3 decode codes
        // [0, GS/2) of each group, warps 4-7 codes [GS/2, GS) (warp-uniform) -----
        const int r = tid & 127;
        const int h = warp >> 2;
        const int row = n0 + r;
        const bool rok = row < p.N;
        const uint8_t *wrow = p.w + (long long)(rok ? row : 0) * p.row_bytes;
        const __half *srow = p.scales + (long long)(rok ? row : 0) * p.G;
        const __half *brow = p.biases ? p.biases + (long long)(rok ? row : 0) * p.G : nullptr;
        // t5: the bytes of this thread's half of the group, from byte FB (0, or
        // 12 / 6 for the second half), NWH words, read as two aligned 16-byte
        // loads (row_bytes is a multiple of 16 here) and realigned in registers.
        // (two-block gs=128: a quarter's bytes start at 0 / 12 for h = 0 and
        // 6 / 18 for h = 1 in even / odd K steps, and span at most 8 bytes)
        constexpr bool Q4 = T5F && GS == 128 && NH == 2;
        constexpr int FB1 = GS == 128 && !Q4 ? 12 : 6;
        constexpr int NWH = GS == 128 && !Q4 ? 4 : 2;
        // 1/2-bit: half h of a K step is HB bytes (HW words) at byte
        // (first code of the step)/CPB + h*HB, one aligned load (row_bytes is
        // a multiple of 2HB and the base is 16-byte aligned)
        constexpr int CPB = FMT == BQD_FMT_AFFINE2 ? 4 : 8;  // codes per byte
        constexpr int HB = KS / (2 * CPB);                   // 4, 8 or 16
        constexpr int HW = T5F ? NWH : HB / 4;               // words decoded per step
        const int fb = h ? FB1 : 0;
        uint4 w0n = make_uint4(0, 0, 0, 0), w1n = make_uint4(0, 0, 0, 0);
        int ow_n = 0;
        uint32_t an[T5F ? 1 : HW];
        uint16_t sb_n = 0, bb_n = 0;
        // the next K step's bytes, scale and bias are requested before the
        // current one is decoded; steps are fetched in order, so the sources
        // advance by one group per call
        long long t5_start = (long long)g_lo * B + fb;
        const uint8_t *wp = wrow + (long long)g_lo * (GS / CPB) + h * HB;
        const __half *sp = srow + g_lo, *bp = brow ? brow + g_lo : nullptr;
        int sstep = 0;  // K steps fetched in the current group (SPG per group)
        int fpar = 0;   // quarters: parity of the K step being fetched
        auto fetch = [&]() {
            if constexpr (T5F) {
                const long long start = t5_start;
                if constexpr (Q4) {
                    t5_start += fpar ? 14 : 12;
                    fpar ^= 1;
                } else {
                    t5_start += B;
                }
                const long long astart = start & ~15LL;
                ow_n = (int)(start & 15);
                w0n = rok ? *reinterpret_cast<const uint4 *>(wrow + astart) : make_uint4(0, 0, 0, 0);
                w1n = rok && astart + 16 < p.row_bytes ? *reinterpret_cast<const uint4 *>(wrow + astart + 16)
                                                       : make_uint4(0, 0, 0, 0);
            } else {
                const uint8_t *src = wp;
                wp += 2 * HB;
                if constexpr (HW == 4) {
                    const uint4 v = rok ? *reinterpret_cast<const uint4 *>(src) : make_uint4(0, 0, 0, 0);
                    an[0] = v.x; an[1] = v.y; an[2] = v.z; an[3] = v.w;
                } else if constexpr (HW == 2) {
                    const uint2 v = rok ? *reinterpret_cast<const uint2 *>(src) : make_uint2(0, 0);
                    an[0] = v.x; an[1] = v.y;
                } else {
                    an[0] = rok ? *reinterpret_cast<const uint32_t *>(src) : 0u;
                }
            }
            sb_n = rok ? __half_as_ushort(*sp) : (uint16_t)0;
            bb_n = rok && bp ? __half_as_ushort(*bp) : (uint16_t)0;
            if constexpr (SPG == 1) {
                ++sp;
                if (bp) ++bp;
            } else if (++sstep == SPG) {
                sstep = 0;
                ++sp;
                if (bp) ++bp;
            }
        };
        // magic exponents: t5 fields sit at bits 2d of both halves; 1/2-bit
        // pair d has its low code at mantissa bit PLO(d), its high one at PHI(d)
        uint32_t mg[5];
#pragma unroll
        for (int d = 0; d < 5; ++d) mg[d] = magic(2 * d) ^ p.zero;
        constexpr int NPAT = FMT == BQD_FMT_AFFINE2 ? 2 : 4;  // 1/2-bit pair patterns per byte
        auto plo = [](int d) { return FMT == BQD_FMT_AFFINE2 ? 4 * d : 2 * d; };
        auto phi = [](int d) { return FMT == BQD_FMT_AFFINE2 ? 4 * d + 2 : 2 * d + 1; };
        uint32_t mgx[NPAT];
#pragma unroll
        for (int d = 0; d < NPAT; ++d)
            mgx[d] = ((magic(plo(d)) & 0xFFFFu) | (magic(phi(d)) & 0xFFFF0000u)) ^ p.zero;
        // this thread's 16-byte chunks of the A tile, relative to the stage
        uint32_t a_off[KS / 16];
#pragma unroll
        for (int q = 0; q < KS / 16; ++q) {
            const int chunk = (KS / 16) * h + q;
            a_off[q] = (uint32_t)((chunk >> 3) * 16384) + sw128_offset(r, chunk & 7);
        }
        int s = 0;          // stage of step it
        uint32_t rpar = 1;  // parity of empty_bar[s] that frees it for step it (>= NST)
        // one K step after its data is in registers: wait for the stage, decode,
        // store the A tile, arrive; false once a bounded wait has expired
        auto step_body = [&](int it, const uint32_t (&cur)[HW], uint16_t sb, uint16_t bb) -> bool {
            if (it >= NST && !wait_bounded(smem_addr(&empty_bar[s]), rpar, p.wait_ns)) {
                abort_flag = 1;
                return false;
            }
            const uint32_t s2 = dup_half(sb), b2 = dup_half(bb);
            // constants -2^(10-p)*s stay finite for |s| < 63; else the exact
            // (magic - offset) * s form is used
            const bool fast = fabsf(__half2float(__ushort_as_half(sb))) < 63.f;
            // this thread's KS/4 words (KS/2 codes, two per word: code 2i low,
            // 2i+1 high): half h of the K step
            uint32_t hv[KS / 4];
            if constexpr (T5F) {
                uint32_t c[5];
#pragma unroll
                for (int d = 0; d < 5; ++d)
                    c[d] = hmul2(s2, dup_half(__half_as_ushort(__float2half_rn(-(float)(1024 >> (2 * d))))));
                auto wv = [&](uint32_t field_word, uint32_t mask, int d) -> uint32_t {
                    const uint32_t hh = (field_word & mask) | mg[d];
                    const uint32_t ts = fast ? hfma2(hh, s2, c[d]) : hmul2(hsub2(hh, mg[d]), s2);  // t*s, exact
                    return hadd2(ts, b2);
                };
                auto lut_of = [&](int j) -> uint32_t {
                    return lut[__byte_perm(cur[j >> 2], 0, 0x4440 | (j & 3)) * kLutCopiesQ +
                               (lane & (kLutCopiesQ - 1))];
                };
                // j below is the byte index within this half's words; codes 5j .. 5j+9
                // of bytes (j, j+1) (relative to the half's first byte)
                auto pair_at = [&](int j, uint32_t *out) {
                    const uint32_t L0 = lut_of(j), L1 = lut_of(j + 1);
                    const uint32_t u = L0 * 16385u;      // fields of byte j, also shifted by 14
                    const uint32_t u2 = L0 + (L1 << 24);  // (trit 4 of byte j, trit 0 of byte j+1) at bit 8
                    const uint32_t u3 = L1 * 16385u;     // fields of byte j+1, also shifted by 14
                    out[0] = wv(u, 0x00030003u, 0);
                    out[1] = wv(u, 0x00300030u, 2);
                    out[2] = wv(u2, 0x03000300u, 4);
                    out[3] = wv(u3, 0x000C000Cu, 1);
                    out[4] = wv(u3, 0x00C000C0u, 3);
                };
                // codes 5j .. 5j+3 of a lone byte j
                auto single_at = [&](int j, uint32_t *out) {
                    const uint32_t u = lut_of(j) * 16385u;
                    out[0] = wv(u, 0x00030003u, 0);
                    out[1] = wv(u, 0x00300030u, 2);
                };
                if (Q4 && (it & 1)) {
                    // odd K step: codes 64..127 of the group.  The four byte pairs
                    // from the fetched byte give codes 60..99 (h = 0, byte 12) or
                    // 90..129 (h = 1, byte 18); the quarter starts at word 2 / 3
                    uint32_t tmp[20];
#pragma unroll
                    for (int jp = 0; jp < 4; ++jp) pair_at(2 * jp, &tmp[5 * jp]);
#pragma unroll
                    for (int i = 0; i < 16; ++i) hv[i] = h ? tmp[i + 3] : tmp[i + 2];
                } else if (GS == 128 && !Q4) {
                    if (h == 0) {  // codes 0..63: byte pairs (0,1) .. (10,11), then byte 12's first four
#pragma unroll
                        for (int jp = 0; jp < 6; ++jp) pair_at(2 * jp, &hv[5 * jp]);
                        single_at(12, &hv[30]);
                    } else {  // codes 64..127: byte pairs (12,13) .. (24,25) give codes 60..129
                        uint32_t tmp[35];
#pragma unroll
                        for (int jp = 0; jp < 7; ++jp) pair_at(2 * jp, &tmp[5 * jp]);  // local bytes 0..13 = group bytes 12..25
#pragma unroll
                        for (int i = 0; i < 32; ++i) hv[i] = tmp[i + 2];
                    }
                } else {
                    // a 64-code group, or the even K step of a two-block gs=128
                    // group (codes 0..63, laid out as a 64-code group's)
                    if (h == 0) {  // codes 0..31: byte pairs (0,1) .. (4,5), then byte 6's first two
                        uint32_t tmp[17];
#pragma unroll
                        for (int jp = 0; jp < 3; ++jp) pair_at(2 * jp, &tmp[5 * jp]);
                        single_at(6, &tmp[15]);
#pragma unroll
                        for (int i = 0; i < 16; ++i) hv[i] = tmp[i];
                    } else {  // codes 32..63: byte pairs (6,7) .. (10,11) give codes 30..59, byte 12 codes 60..63
                        uint32_t tmp[15];
#pragma unroll
                        for (int jp = 0; jp < 3; ++jp) pair_at(2 * jp, &tmp[5 * jp]);  // local bytes 0..6 = group bytes 6..12
#pragma unroll
                        for (int i = 0; i < 14; ++i) hv[i] = tmp[i + 1];
                        single_at(6, &hv[14]);
                    }
                }
            } else {
                uint32_t c[NPAT];
#pragma unroll
                for (int d = 0; d < NPAT; ++d) {
                    const uint32_t off = (uint32_t)__half_as_ushort(__float2half_rn(-(float)(1024 >> plo(d)))) |
                                         ((uint32_t)__half_as_ushort(__float2half_rn(-(float)(1024 >> phi(d)))) << 16);
                    c[d] = hmul2(s2, off);
                }
                // byte y of word q holds codes CPB*(4q+y) ..; it is copied into both
                // 16-bit halves, and pattern d takes the low half's code at bit
                // PLO(d) and the high half's at PHI(d) (pair 2-bit: codes 4y+2d,
                // 4y+2d+1; 1-bit: codes 8y+2d, 8y+2d+1)
#pragma unroll
                for (int q = 0; q < HW; ++q)
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        const uint32_t dup = __byte_perm(cur[q], 0, 0x4040u | (uint32_t)y | ((uint32_t)y << 8));
#pragma unroll
                        for (int d = 0; d < NPAT; ++d) {
                            const uint32_t mask = (1u << plo(d)) * (CPB == 4 ? 3u : 1u) |
                                                  ((1u << phi(d)) * (CPB == 4 ? 3u : 1u)) << 16;
                            const uint32_t hh = (dup & mask) | mgx[d];
                            const uint32_t qs = fast ? hfma2(hh, s2, c[d]) : hmul2(hsub2(hh, mgx[d]), s2);
                            hv[(CPB / 2) * (4 * q + y) + d] = hadd2(qs, b2);
                        }
                    }
            }
            // store into the stage's A tile (K-major, 128-byte swizzle): 16-byte
            // chunk q of this half is chunk (KS/16) h + q of the row.  Rows past
            // N decode to zeros: their bytes, scale and bias were loaded as 0.
            const uint32_t at = smem_addr(smem + (size_t)s * stage_bytes);
#pragma unroll
            for (int q = 0; q < KS / 16; ++q)
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(at + a_off[q]), "r"(hv[4 * q]),
                             "r"(hv[4 * q + 1]), "r"(hv[4 * q + 2]), "r"(hv[4 * q + 3])
                             : "memory");
            fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
            mbar_arrive(smem_addr(&a_full[s]));
            if (++s == NST) {
                s = 0;
                rpar ^= 1u;
            }
            return true;
        };
        if constexpr (NH == 2 && !T5F) {
            // 64-code steps are short: two steps of bytes, scale and bias are in
            // flight per thread, in two register slots used alternately (two
            // steps per iteration, so the slot of each load is a constant).
            // Loads are unconditional: past the last step the sources stop
            // advancing and the extra fetch re-reads it (valid memory, unused).
            uint32_t anq[2][HW];
            uint16_t sbq[2], bbq[2];
            int fetched = 0;
            auto fetch_into = [&](auto U) {
                constexpr int u = decltype(U)::value;
                const bool adv = ++fetched < steps;
                const uint8_t *src = wp;
                wp += adv ? 2 * HB : 0;
                if constexpr (HW == 2) {
                    const uint2 v = rok ? *reinterpret_cast<const uint2 *>(src) : make_uint2(0, 0);
                    anq[u][0] = v.x;
                    anq[u][1] = v.y;
                } else {
                    anq[u][0] = rok ? *reinterpret_cast<const uint32_t *>(src) : 0u;
                }
                sbq[u] = rok ? __half_as_ushort(*sp) : (uint16_t)0;
                bbq[u] = rok && bp ? __half_as_ushort(*bp) : (uint16_t)0;
                int gadv = adv ? 1 : 0;
                if constexpr (SPG > 1) {
                    sstep += gadv;
                    gadv = sstep == SPG ? 1 : 0;
                    sstep = gadv ? 0 : sstep;
                }
                sp += gadv;
                if (bp) bp += gadv;
            };
            if (steps > 0) {
                fetch_into(std::integral_constant<int, 0>{});
                fetch_into(std::integral_constant<int, 1>{});
            }
            bool stop = false;
            for (int it0 = 0; it0 < steps && !stop; it0 += 2) {
                auto one = [&](auto U) {
                    constexpr int u = decltype(U)::value;
                    const int it = it0 + u;
                    if (stop || it >= steps) return;
                    uint32_t cur[HW];
#pragma unroll
                    for (int q = 0; q < HW; ++q) cur[q] = anq[u][q];
                    const uint16_t sb = sbq[u];
                    const uint16_t bb =
                        rok ? (brow ? bbq[u] : __half_as_ushort(sym_bias(__ushort_as_half(sb), p.ratio))) : (uint16_t)0;
                    fetch_into(U);
                    if (!step_body(it, cur, sb, bb)) stop = true;
                };
                one(std::integral_constant<int, 0>{});
                one(std::integral_constant<int, 1>{});
            }
        } else {
            if (steps > 0) fetch();
            for (int it = 0; it < steps; ++it) {
                uint32_t cur[HW];
                if constexpr (T5F) {
                    const uint32_t W[8] = {w0n.x, w0n.y, w0n.z, w0n.w, w1n.x, w1n.y, w1n.z, w1n.w};
                    const int wo = ow_n >> 2, sh = (ow_n & 3) * 8;
                    uint32_t V[NWH + 1];
#pragma unroll
                    for (int i = 0; i <= NWH; ++i) {
                        const uint32_t lo = (wo & 1) ? W[i + 1] : W[i];
                        const uint32_t hi = (wo & 1) ? W[i + 3] : W[i + 2];
                        V[i] = (wo & 2) ? hi : lo;
                    }
#pragma unroll
                    for (int q = 0; q < NWH; ++q) cur[q] = __funnelshift_r(V[q], V[q + 1], sh);
                } else {
#pragma unroll
                    for (int q = 0; q < HW; ++q) cur[q] = an[q];
                }
                const uint16_t sb = sb_n;
                const uint16_t bb = rok ? (brow ? bb_n : __half_as_ushort(sym_bias(__ushort_as_half(sb), p.ratio)))
                                        : (uint16_t)0;
                if (it + 1 < steps) fetch();
                if (!step_body(it, cur, sb, bb)) break;
            }
        }
    }

    // ---- epilogue: warp w drains TMEM lanes 32 (w % 4) .. +31, column half w / 4 ------
    __syncthreads();
    // every issued MMA has completed before TMEM is read or freed
    if (warp < kDecodeWarpsQ && steps > 0) wait_bounded(smem_addr(&done_bar), 0, kDrainWaitNs);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool ok_all = !abort_flag;
    // split K: a reduce-scatter over 32-column blocks.  Rank q owns blocks
    // [q nb / S, (q+1) nb / S) and writes their outputs; every other rank
    // stores its partials of those blocks into q's stage ring, laid out
    // [S-1 sources][128 rows][W_q + 4] fp32 (a row padded by 16 bytes, so that
    // the lanes' 16-byte accesses spread over the banks), and q adds the S
    // partials in rank order.
    const int nb = C / 32;
    const int lo_me = rank * nb / S, hi_me = (rank + 1) * nb / S;
    const int wst_me = (hi_me - lo_me) * 32 + 4;
    float *red = reinterpret_cast<float *>(smem);
    if (S > 1) cluster_sync();  // every rank's MMAs are complete: the rings are free
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int row = n0 + r;
    // columns of this warp: half (warp >> 2) of bx, in blocks of 32 (bx = 32: warps 0-3 only)
    const int cw = C >= 64 ? C / 2 : C;
    const int c_beg = C >= 64 ? (warp >> 2) * cw : 0;
    const bool drains = warp < kDecodeWarpsQ && (C >= 64 || warp < 4);
    if (drains && S > 1 && steps > 0) {
        for (int c0 = c_beg; c0 < c_beg + cw; c0 += 32) {
            const int b = c0 >> 5;
            int q = 0;
            while ((q + 1) * nb / S <= b) ++q;  // the owner: lo_q <= b < hi_q
            if (q == rank) continue;
            const int lo_q = q * nb / S, hi_q = (q + 1) * nb / S;
            const int wst = (hi_q - lo_q) * 32 + 4;
            const int slot = rank < q ? rank : rank - 1;
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)c0, v);
            const uint32_t dst = smem_addr(red + ((size_t)slot * 128 + r) * wst + (b - lo_q) * 32);
#pragma unroll
            for (int j = 0; j < 32; j += 4) st_cluster_v4(dst + 4 * j, (uint32_t)q, v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (S > 1) cluster_sync();
    if (drains && ok_all) {
        for (int c0 = c_beg; c0 < c_beg + cw; c0 += 32) {
            const int b = c0 >> 5;
            if (b < lo_me || b >= hi_me) continue;
            uint32_t v[32];
            if (steps > 0) {
                tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)c0, v);
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = 0u;
            }
            float acc[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = 0.f;
            for (int src = 0; src < S; ++src) {
                if (src == rank) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) acc[q] += __uint_as_float(v[q]);
                } else if (src * p.gpr < p.G) {  // ranks without groups sent nothing
                    const int slot = src < rank ? src : src - 1;
                    const float *rp = red + ((size_t)slot * 128 + r) * wst_me + (b - lo_me) * 32;
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(rp + q);
                        acc[q] += t4.x;
                        acc[q + 1] += t4.y;
                        acc[q + 2] += t4.z;
                        acc[q + 3] += t4.w;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int m = m0 + c0 + q;
                if (row < p.N && m < p.M) p.out[(size_t)m * p.N + row] = __float2half_rn(acc[q]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpQ) tmem_dealloc(tmem, (uint32_t)C);
}

template <int GS, int NH>
__global__ void __launch_bounds__(kThreadsQ, 1)
qmm_t5_kernel(const __grid_constant__ CUtensorMap xmap, const QmmParams p)
{
    qmm_body<BQD_FMT_T5, GS, NH>(xmap, p);
}

template <int FMT, int GS, int NH>
__global__ void __launch_bounds__(kThreadsQ, 1)
qmm_affine_kernel(const __grid_constant__ CUtensorMap xmap, const QmmParams p)
{
    qmm_body<FMT, GS, NH>(xmap, p);
}

// ---- host side -------------------------------------------------------------------

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

using QmmKernel = void (*)(const CUtensorMap, const QmmParams);

// clusters of S CTAs (CTAs for S = 1) that can be resident at once
int qmm_slots(QmmKernel kern, int S, size_t smem)
{
    struct Entry { int dev; QmmKernel kern; int S; size_t smem; int slots; };
    static Entry cache[64];
    static int n = 0;
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].dev == dev && cache[i].kern == kern && cache[i].S == S && cache[i].smem == smem) return cache[i].slots;
    int slots = 0;
    if (S == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreadsQ, smem) == cudaSuccess)
            slots = per_sm * sm_count();
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(S * 16);
        cfg.blockDim = dim3(kThreadsQ);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = S;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&slots, kern, &cfg) != cudaSuccess) slots = 0;
    }
    cudaGetLastError();
    if (n < 64) cache[n++] = Entry{dev, kern, S, smem, slots};
    return slots;
}

template <int FMT, int GS, int NH>
int launch_gs(QmmParams p, const CUtensorMap &map, int tiles, size_t per_stage, int cols, cudaStream_t s)
{
    QmmKernel kern;
    if constexpr (FMT == BQD_FMT_T5)
        kern = qmm_t5_kernel<GS, NH>;
    else
        kern = qmm_affine_kernel<FMT, GS, NH>;
    static int configured_dev[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured_dev[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQmmSmemMax) != cudaSuccess)
            return BQD_ERR_CUDA;
        configured_dev[dev] = 1;
    }
    const size_t smem = (size_t)p.stages * per_stage + 1024;
    // Split K over a cluster of S CTAs while every cluster of the grid is
    // resident at once (occupancy query), each rank keeps >= 4 groups, and the
    // partials a rank receives fit its stage ring.  (A split that needs more
    // than one wave measured slower: narrow layers at M = 512 and 2048 lost
    // 0-10% with S = 4-5 over two or three waves against S = 1.)
    const int nb = cols / 32;
    int bestS = 1;
    for (int S = 2; S <= 8; ++S) {
        if (p.G < 4 * S) break;
        int wmax = 0;
        for (int q = 0; q < S; ++q) wmax = std::max(wmax, ((q + 1) * nb / S - q * nb / S) * 32);
        if ((size_t)(S - 1) * 128 * (wmax + 4) * 4 > (size_t)p.stages * per_stage) break;
        if (tiles > qmm_slots(kern, S, smem)) break;
        bestS = S;
    }
    p.S = bestS;
    p.gpr = (p.G + bestS - 1) / bestS;
    if (opt_debug_plan())
        fprintf(stderr, "bqd qmm plan: fmt=%d M=%d N=%d K=%d gs=%d -> bx=%d x%d tiles=%d S=%d gpr=%d stages=%d smem=%zu\n",
                FMT, p.M, p.N, p.K, GS, p.bx, NH, tiles, p.S, p.gpr, p.stages, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * p.S);
    cfg.blockDim = dim3(kThreadsQ);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p.S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, map, p) == cudaSuccess ? BQD_OK : BQD_ERR_CUDA;
}

}  // namespace

int take_qmm_timeouts(unsigned int *count)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmm_timeouts, sizeof(v)) != cudaSuccess) return BQD_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_qmm_timeouts, &zero, sizeof(zero)) != cudaSuccess) return BQD_ERR_CUDA;
    *count = v;
    return BQD_OK;
}

int launch_qmm(const QmvArgs &a, cudaStream_t s)
{
    // the decode reads 16-byte aligned pieces of each t5 row; a 1/2-bit half
    // group is 4, 8 or 16 bytes at a multiple of its size (row_bytes = G * gs/4
    // or G * gs/8), aligned once the base is
    if (a.fmt == BQD_FMT_T5 && a.row_bytes % 16 != 0) return BQD_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(a.w) & 15) return BQD_ERR_UNSUPPORTED;
    if (a.K > (int64_t)1 << 30 || a.N > (int64_t)1 << 30 || a.M > (int64_t)1 << 30) return BQD_ERR_UNSUPPORTED;
    auto enc = encode_fn();
    if (!enc) return BQD_ERR_UNSUPPORTED;
    QmmParams p;
    p.w = a.w; p.scales = a.scales; p.biases = a.biases; p.out = a.out; p.ratio = a.ratio;
    p.M = (int)a.M; p.N = (int)a.N; p.K = (int)a.K; p.G = (int)a.G;
    p.row_bytes = a.row_bytes;
    p.wait_ns = (unsigned long long)opt_wait_ns();
    p.zero = 0;
    p.bx = a.M <= 32 ? 32 : (a.M <= 64 ? 64 : (a.M <= 128 ? 128 : 256));
    // more than 256 x rows on a wide layer: two 256-column blocks per CTA (the
    // decoded weight tile serves 512 columns), K steps of 64 codes.  Narrow
    // layers keep one block: their few 128-row tiles would leave SMs idle
    // (measured: down projection, M=512, 813 -> 470 TFLOP/s)
    const bool pair = a.M > 256 && a.N >= 8192;
    const int NH = pair ? 2 : 1;
    const int KS = pair ? 64 : a.gs;
    const int cols = NH * p.bx;
    const int n_tiles = (p.N + 127) / 128, m_tiles = (p.M + cols - 1) / cols;
    const int tiles = n_tiles * m_tiles;
    const size_t per_stage = (size_t)128 * KS * 2 + (size_t)cols * KS * 2;
    p.stages = (int)((kQmmSmemMax - 1024) / per_stage);
    if (p.stages > kMaxStagesQ) p.stages = kMaxStagesQ;
    if (p.stages < 2) return BQD_ERR_UNSUPPORTED;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)p.bx};
    cuuint32_t estr[2] = {1, 1};
    CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(a.x), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return BQD_ERR_CUDA;
    if (a.fmt == BQD_FMT_T5) {
        if (pair)
            return a.gs == 64 ? launch_gs<BQD_FMT_T5, 64, 2>(p, map, tiles, per_stage, cols, s)
                              : launch_gs<BQD_FMT_T5, 128, 2>(p, map, tiles, per_stage, cols, s);
        return a.gs == 64 ? launch_gs<BQD_FMT_T5, 64, 1>(p, map, tiles, per_stage, cols, s)
                          : launch_gs<BQD_FMT_T5, 128, 1>(p, map, tiles, per_stage, cols, s);
    }
    if (a.fmt == BQD_FMT_AFFINE2) {
        if (pair)
            return a.gs == 64 ? launch_gs<BQD_FMT_AFFINE2, 64, 2>(p, map, tiles, per_stage, cols, s)
                              : launch_gs<BQD_FMT_AFFINE2, 128, 2>(p, map, tiles, per_stage, cols, s);
        return a.gs == 64 ? launch_gs<BQD_FMT_AFFINE2, 64, 1>(p, map, tiles, per_stage, cols, s)
                          : launch_gs<BQD_FMT_AFFINE2, 128, 1>(p, map, tiles, per_stage, cols, s);
    }
    if (pair)
        return a.gs == 64 ? launch_gs<BQD_FMT_AFFINE1, 64, 2>(p, map, tiles, per_stage, cols, s)
                          : launch_gs<BQD_FMT_AFFINE1, 128, 2>(p, map, tiles, per_stage, cols, s);
    return a.gs == 64 ? launch_gs<BQD_FMT_AFFINE1, 64, 1>(p, map, tiles, per_stage, cols, s)
                      : launch_gs<BQD_FMT_AFFINE1, 128, 1>(p, map, tiles, per_stage, cols, s);
}

}  // namespace bqd
