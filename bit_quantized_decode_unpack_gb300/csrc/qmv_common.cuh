// Device helpers shared by the tensor-core QMV kernels (inline PTX wrappers for
// fp16x2 arithmetic, mma.sync, streaming loads, mbarriers, bulk copies,
// clusters and programmatic dependent launch).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace bqd {
namespace qmvdev {

// warps per CTA of the tensor-core QMV kernels
constexpr int kWarps = 8;

// ---- PTX helpers -------------------------------------------------------------

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// (a & MASK) | c in one LOP3, MASK an immediate, c a register
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}




__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, uint32_t rank, float v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ uint32_t dup_half(uint16_t h) { return (uint32_t)h | ((uint32_t)h << 16); }

// fp16 bits of a value 2^(10-p) + q whose code field q sits at mantissa bit p
__host__ __device__ constexpr uint32_t magic(int p) { return (uint32_t)((25 - p) << 10) * 0x00010001u; }

// mbarrier try_wait (non-blocking probe of a phase)
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// order earlier generic-proxy accesses of shared memory before later
// async-proxy (bulk copy) writes to it
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- bounded waits ----------------------------------------------------------------

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// non-blocking probe of a phase (never suspends the thread)
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` of the mbarrier at `bar`; give up
// once `limit_ns` of %globaltimer have passed, counting the expiry in *expired.
// Limits of at least 20 us probe with try_wait (which may suspend the thread
// for a while) and read the clock every 64 probes; shorter ones spin on
// test_wait (a try_wait may sleep until the phase completes, which would hide
// a short limit).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                                              unsigned int *expired)
{
    if (limit_ns >= 20000ull) {
        if (mbar_try_wait(bar, parity)) return true;
        const unsigned long long t0 = globaltimer_ns();
        while (true) {
            for (int i = 0; i < 64; ++i)
                if (mbar_try_wait(bar, parity)) return true;
            if (globaltimer_ns() - t0 >= limit_ns) break;
        }
    } else {
        if (mbar_test_wait(bar, parity)) return true;
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < limit_ns)
            if (mbar_test_wait(bar, parity)) return true;
    }
    atomicAdd(expired, 1u);
    return false;
}

// limit of the waits that let a CTA's own copies (and MMAs) finish before it
// leaves: they always keep the full second
constexpr unsigned long long kDrainWaitNs = 1000000000ull;

__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_u16(const __half *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_stream_v4_if(const void *p, bool pred)
{
    uint4 v;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "@q ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "r"((int)pred));
    return v;
}

__device__ __forceinline__ uint2 ld_stream_v2_if(const void *p, bool pred)
{
    uint2 v;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\t"
        "@q ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];\n\t}"
        : "=r"(v.x), "=r"(v.y)
        : "l"(p), "r"((int)pred));
    return v;
}

__device__ __forceinline__ uint32_t ld_u32_if(const void *p, bool pred)
{
    uint32_t v;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\tmov.b32 %0, 0;\n\t@q ld.global.nc.u32 %0, [%1];\n\t}"
        : "=r"(v)
        : "l"(p), "r"((int)pred));
    return v;
}

__device__ __forceinline__ uint16_t ld_u16_if(const __half *p, bool pred)
{
    uint16_t v;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\tmov.b16 %0, 0;\n\t@q ld.global.nc.u16 %0, [%1];\n\t}"
        : "=h"(v)
        : "l"(p), "r"((int)pred));
    return v;
}


// Position of one warp in its unit sequence u = warp, warp+8, ... (tile-major;
// a unit is 16 weight rows x one 256-code chunk).
struct UnitPos {
    int tl, cl;
    __device__ __forceinline__ void start(int warp, int ncl)
    {
        tl = 0;
        cl = warp;
        while (cl >= ncl) {
            cl -= ncl;
            ++tl;
        }
    }
    // returns the number of row tiles crossed
    __device__ __forceinline__ int advance(int ncl)
    {
        int crossed = 0;
        cl += kWarps;
        while (cl >= ncl) {
            cl -= ncl;
            ++crossed;
        }
        tl += crossed;
        return crossed;
    }
};

}  // namespace qmvdev
}  // namespace bqd
