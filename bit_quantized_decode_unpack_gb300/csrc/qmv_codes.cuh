// Code-unpack traits shared by the 1/2-bit tensor-core decode kernels.
//
// A 256-code chunk of one weight row is turned into fp16x2 MMA A registers
// with one LOP3 per two codes: the code lands at mantissa bit p of an fp16
// whose exponent makes its value 2^(10-p) + q (page "oMLX Bonsai 自定义内核:
// Qwen 系列快速 QMV 路径完整解析", §二.1: codes are unpacked in registers, no
// floating-point weight matrix is materialised).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "bqd.h"
#include "qmv_common.cuh"

namespace bqd {
namespace qmvdev {

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

}  // namespace qmvdev
}  // namespace bqd
