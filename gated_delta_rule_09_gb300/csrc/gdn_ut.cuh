// Blocked forward substitution for the UT transform of one 64-token chunk,
// shared by the tcgen05 producer and the standalone batched inverse.
//
// T = (I + A)^{-1} for a strictly lower 64 x 64 A ("RNN的复兴03：现代RNN的并行计算",
// §2.3.1: the column recursion T[i,j] = -sum_{m=j}^{i-1} A[i,m] T[m,j], here
// with the sign of "从零开始的 GDN 推导", §"UT transform"), applied to blocks:
// (1) the four 16 x 16 diagonal blocks by forward substitution, half a warp
//     per block and a lane per column, in registers;
// (2) 16 -> 32: T[1,0] = -T11 (A10 T00) for the block pairs (0,1), (2,3);
// (3) 32 -> 64: T[32:64, 0:32] = -T2 (A21 T1).
// In place: A and T share `As` (fp32, row stride kUtLd); every block of A is
// dead before the same block of T is written, and A's zero upper triangle is
// exactly the zero upper blocks the merges read, so the loops need no
// triangular bounds; the second product of each merge still stops at the
// last row a warp owns, since the lower-triangular left factor is exactly
// zero beyond it (the sums are unchanged, bit for bit).  `Xs` is merge scratch of 32 x kUtLdX3 floats.  128 threads (t =
// 0..127, four whole warps) synchronise on named barrier `bar_id`.
#pragma once

#include <stdint.h>

#include "sm100_ptx.cuh"

namespace gdn_ut {

constexpr int kUtLd = 68;     // fp32 row stride of A / T: 16-byte rows, 4-bank offset per row
constexpr int kUtLdX2 = 20;   // row stride of the 16x16 merge scratch
constexpr int kUtLdX3 = 36;   // row stride of the 32x32 merge scratch

// (1) the four 16 x 16 diagonal blocks, in place, on warps 0-1: lane l of
// warp w owns column l & 15 of block 2w + (l >> 4) and substitutes forward
// down the rows (warps 2-3 pass through; the caller synchronises after it).
__device__ __forceinline__ void ut_diag16(float *As, int t)
{
    float *Ts = As;
    const int lane = t & 31, quad = t >> 5;
    constexpr int kLdA = kUtLd;
    if (quad < 2) {
        const int b = 2 * quad + (lane >> 4), l = lane & 15;
        float tv[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) tv[r] = (r == l) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m)
                if (m >= l) acc = fmaf(As[(16 * b + r) * kLdA + 16 * b + m], tv[m], acc);
            if (r > l) tv[r] = -acc;
        }
        __syncwarp();  // every lane has read its A block before T overwrites it
#pragma unroll
        for (int r = 0; r < 16; ++r) Ts[(16 * b + r) * kLdA + 16 * b + l] = tv[r];
    }
}

__device__ __forceinline__ void ut_inverse_64(float *As, float *Xs, int t, uint32_t bar_id)
{
    using namespace sm100;
    float *Ts = As;
    const int quad = t >> 5;
    constexpr int kLdA = kUtLd, kLdX2 = kUtLdX2, kLdX3 = kUtLdX3;
    ut_diag16(As, t);
    named_sync(bar_id, 128);
    // (2) 16 -> 32: T[1,0] = -T11 (A10 T00) for the block pairs (0,1), (2,3).
    //     64 threads per pair, each a 1x4 block of the 16x16 result with
    //     independent accumulators; the never-written upper blocks of T
    //     are zero, so every loop has fixed bounds.
    {
        const int pp = t >> 6, r = (t & 63) >> 2, c4 = (t & 3) * 4;
        const int R = 16 * (2 * pp + 1), Cc = 32 * pp;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2  // partial unrolling: the compact loop stays in the instruction cache
        for (int m = 0; m < 16; ++m) {
            const float av = As[(R + r) * kLdA + Cc + m];
            const float4 tv = *reinterpret_cast<const float4 *>(Ts + (Cc + m) * kLdA + Cc + c4);
            acc.x = fmaf(av, tv.x, acc.x);
            acc.y = fmaf(av, tv.y, acc.y);
            acc.z = fmaf(av, tv.z, acc.z);
            acc.w = fmaf(av, tv.w, acc.w);
        }
        *reinterpret_cast<float4 *>(Xs + pp * 16 * kLdX2 + r * kLdX2 + c4) = acc;
        named_sync(bar_id, 128);
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        // T11 is lower triangular: this warp's rows r stay below mend2
        const int mend2 = 8 * ((quad & 1) + 1);
#pragma unroll 2
        for (int m = 0; m < mend2; ++m) {
            const float tv = Ts[(R + r) * kLdA + R + m];
            const float4 xv = *reinterpret_cast<const float4 *>(Xs + pp * 16 * kLdX2 + m * kLdX2 + c4);
            acc.x = fmaf(tv, xv.x, acc.x);
            acc.y = fmaf(tv, xv.y, acc.y);
            acc.z = fmaf(tv, xv.z, acc.z);
            acc.w = fmaf(tv, xv.w, acc.w);
        }
        *reinterpret_cast<float4 *>(Ts + (R + r) * kLdA + Cc + c4) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    named_sync(bar_id, 128);
    // (3) 32 -> 64: T[32:64, 0:32] = -T2 (A21 T1); each thread a 2x4 block.
    {
        const int r2 = (t >> 3) * 2, c4 = (t & 7) * 4;
        float4 a0c = make_float4(0.f, 0.f, 0.f, 0.f), a1c = a0c;
#pragma unroll 2
        for (int m = 0; m < 32; ++m) {
            const float a0 = As[(32 + r2) * kLdA + m], a1 = As[(33 + r2) * kLdA + m];
            const float4 tv = *reinterpret_cast<const float4 *>(Ts + m * kLdA + c4);
            a0c.x = fmaf(a0, tv.x, a0c.x); a0c.y = fmaf(a0, tv.y, a0c.y);
            a0c.z = fmaf(a0, tv.z, a0c.z); a0c.w = fmaf(a0, tv.w, a0c.w);
            a1c.x = fmaf(a1, tv.x, a1c.x); a1c.y = fmaf(a1, tv.y, a1c.y);
            a1c.z = fmaf(a1, tv.z, a1c.z); a1c.w = fmaf(a1, tv.w, a1c.w);
        }
        *reinterpret_cast<float4 *>(Xs + r2 * kLdX3 + c4) = a0c;
        *reinterpret_cast<float4 *>(Xs + (r2 + 1) * kLdX3 + c4) = a1c;
        named_sync(bar_id, 128);
        a0c = make_float4(0.f, 0.f, 0.f, 0.f);
        a1c = a0c;
        const int mend3 = 8 * (quad + 1);  // T2 is lower: this warp's rows are below mend3
#pragma unroll 2
        for (int m = 0; m < mend3; ++m) {
            const float t0 = Ts[(32 + r2) * kLdA + 32 + m], t1 = Ts[(33 + r2) * kLdA + 32 + m];
            const float4 xv = *reinterpret_cast<const float4 *>(Xs + m * kLdX3 + c4);
            a0c.x = fmaf(t0, xv.x, a0c.x); a0c.y = fmaf(t0, xv.y, a0c.y);
            a0c.z = fmaf(t0, xv.z, a0c.z); a0c.w = fmaf(t0, xv.w, a0c.w);
            a1c.x = fmaf(t1, xv.x, a1c.x); a1c.y = fmaf(t1, xv.y, a1c.y);
            a1c.z = fmaf(t1, xv.z, a1c.z); a1c.w = fmaf(t1, xv.w, a1c.w);
        }
        *reinterpret_cast<float4 *>(Ts + (32 + r2) * kLdA + c4) =
            make_float4(-a0c.x, -a0c.y, -a0c.z, -a0c.w);
        *reinterpret_cast<float4 *>(Ts + (33 + r2) * kLdA + c4) =
            make_float4(-a1c.x, -a1c.y, -a1c.z, -a1c.w);
    }
    named_sync(bar_id, 128);
}

}  // namespace gdn_ut
