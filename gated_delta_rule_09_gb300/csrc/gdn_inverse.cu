// Batched UT inverse T = (I + A)^{-1} for strictly lower C x C matrices A
// (C <= 64, zero-padded to 64: the padding block of T is the identity), by
// two methods, for comparison:
//
//  method 0, blocked forward substitution on CUDA cores (fp32): the routine
//    the tcgen05 producer runs per chunk (gdn_ut.cuh), one 128-thread CTA per
//    matrix.
//  method 1, the nilpotent doubling product on tcgen05 tensor cores.  A is
//    strictly lower, so A^64 = 0 and the Neumann series of
//    "RNN的复兴03：现代RNN的并行计算" (§2.3.2) is finite:
//        (I + A)^{-1} = sum_{n<64} (-A)^n
//                     = (I - A)(I + A^2)(I + A^4)(I + A^8)(I + A^16)(I + A^32).
//    Five squarings X_k = X_{k-1}^2 (X_0 = -A, fp16 operands, fp32 in TMEM)
//    and five products Q_k = Q_{k-1} + Q_{k-1} X_k accumulated in fp32 in
//    TMEM onto Q_{k-1} itself (Q_0 = I - A), so only the correction term
//    carries fp16 operand rounding.  The squaring for k + 1 and the product
//    for k both read X_k and are issued together: six MMA round trips per
//    matrix.  One row-major 128-byte-swizzled fp16 tile serves as the
//    K-major A operand and as the MN-major B operand.  M = 64: row 16q + r
//    of a result sits in TMEM lane 32q + r, read by lane r < 16 of warp q.
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_internal.h"
#include "gdn_ut.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace sm100;

constexpr int kN = 64;
constexpr uint64_t kWaitNs = 2000000000ull;

// ---------------------------------------------------------------- method 0
__global__ void __launch_bounds__(128) gdn_inv_fs_kernel(const float *__restrict__ A,
                                                         float *__restrict__ T, int C)
{
    __shared__ __align__(16) float As[kN * gdn_ut::kUtLd];
    __shared__ __align__(16) float Xs[32 * gdn_ut::kUtLdX3];
    const int t = threadIdx.x;
    const size_t base = (size_t)blockIdx.x * C * C;
    for (int idx = t; idx < kN * kN; idx += 128) {
        const int i = idx >> 6, j = idx & 63;
        As[i * gdn_ut::kUtLd + j] = (j < i && i < C) ? A[base + (size_t)i * C + j] : 0.f;
    }
    __syncthreads();
    gdn_ut::ut_inverse_64(As, Xs, t, 1);
    for (int idx = t; idx < C * C; idx += 128) {
        const int i = idx / C, j = idx % C;
        T[base + idx] = As[i * gdn_ut::kUtLd + j];
    }
}

// ---------------------------------------------------------------- method 1
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Row `i` (64 values) into a row-major fp16 swizzled tile.
__device__ __forceinline__ void store_row(uint8_t *tile, int i, const float *x)
{
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 u = make_uint4(pack2(x[8 * c], x[8 * c + 1]), pack2(x[8 * c + 2], x[8 * c + 3]),
                             pack2(x[8 * c + 4], x[8 * c + 5]), pack2(x[8 * c + 6], x[8 * c + 7]));
        *reinterpret_cast<uint4 *>(tile + sw128(i, c)) = u;
    }
}

// D (+)= X Y for 64 x 64 tiles X (K-major) and Y (MN-major), both row-major.
__device__ __forceinline__ void mma64(uint32_t d, const uint8_t *x, const uint8_t *y, bool acc)
{
    const uint32_t id = idesc_f16_f32(64, 64, 0, 1);
    const uint64_t dx = sdesc_sw128(smem_u32(x), 16, 1024);
    const uint64_t dy = sdesc_sw128(smem_u32(y), 8192, 1024);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
        mma_f16kind(d, dx + ks * (32 >> 4), dy + ks * (2048 >> 4), id, acc || ks > 0);
}

__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, unsigned int *status)
{
    if (mbar_wait(bar, parity, kWaitNs)) return true;
    atomicOr(status, 0x2u);
    return false;
}

__global__ void __launch_bounds__(128, 4) gdn_inv_tc_kernel(const float *__restrict__ A,
                                                            float *__restrict__ T, int C,
                                                            unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *X[2] = {sm, sm + 8192};   // X_{k} tiles, double-buffered
    uint8_t *Qt = sm + 16384;          // fp16 copy of Q_{k-1}
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + 24576);
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + 24576 + 64);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int i = 16 * warp + lane;    // the row this lane owns (lanes < 16)
    const bool owner = lane < 16;
    const size_t base = (size_t)blockIdx.x * C * C;

    if (warp == 0) {
        tmem_alloc(slot, 128);
        tmem_relinquish();
    }
    if (t == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // Q_0 = I - A (fp32 into TMEM, fp16 tile) and X_0 = -A (fp16 tile)
    float x[64];
#pragma unroll
    for (int j = 0; j < 64; ++j)
        x[j] = (owner && j < i && i < C && j < C) ? -A[base + (size_t)i * C + j] : 0.f;
    if (owner) store_row(X[0], i, x);
#pragma unroll
    for (int j = 0; j < 64; ++j) x[j] += (owner && j == i) ? 1.f : 0.f;
    if (owner) store_row(Qt, i, x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot, dp = tb, dq = tb + 64;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    tmem_st32(dq + lane_base, *reinterpret_cast<float(*)[32]>(x));
    tmem_st32(dq + lane_base + 32, *reinterpret_cast<float(*)[32]>(x + 32));
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // every wait is bounded and every thread runs every step, so the
    // barriers below are reached by all threads even after a timeout
    uint32_t phase = 0;
    bool ok = true;
    // X_1 = X_0^2
    if (t == 0) {
        tc_fence_after();
        mma64(dp, X[0], X[0], false);
        mma_commit(bar);
    }
    ok = wait_bounded(bar, phase, status) && ok;
    phase ^= 1;
    tc_fence_after();
    tmem_ld32(dp + lane_base, *reinterpret_cast<float(*)[32]>(x));
    tmem_ld32(dp + lane_base + 32, *reinterpret_cast<float(*)[32]>(x + 32));
    tmem_ld_wait();
    if (owner) store_row(X[1], i, x);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    for (int k = 1; k <= 5; ++k) {
        // Q_k = Q_{k-1} + Q_{k-1} X_k;  X_{k+1} = X_k^2
        if (t == 0) {
            tc_fence_after();
            mma64(dq, Qt, X[k & 1], true);
            if (k < 5) mma64(dp, X[k & 1], X[k & 1], false);
            mma_commit(bar);
        }
        ok = wait_bounded(bar, phase, status) && ok;
        phase ^= 1;
        tc_fence_after();
        if (k < 5) {
            tmem_ld32(dq + lane_base, *reinterpret_cast<float(*)[32]>(x));
            tmem_ld32(dq + lane_base + 32, *reinterpret_cast<float(*)[32]>(x + 32));
            tmem_ld_wait();
            if (owner) store_row(Qt, i, x);
            tmem_ld32(dp + lane_base, *reinterpret_cast<float(*)[32]>(x));
            tmem_ld32(dp + lane_base + 32, *reinterpret_cast<float(*)[32]>(x + 32));
            tmem_ld_wait();
            if (owner) store_row(X[(k + 1) & 1], i, x);
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
        }
    }
    // T = Q_5
    tmem_ld32(dq + lane_base, *reinterpret_cast<float(*)[32]>(x));
    tmem_ld32(dq + lane_base + 32, *reinterpret_cast<float(*)[32]>(x + 32));
    tmem_ld_wait();
    if (owner && i < C && ok) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
            if (j < C) T[base + (size_t)i * C + j] = x[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 128);
    }
}

}  // namespace

cudaError_t gdn_launch_ut_inverse(const float *A, float *T, int count, int C, int method,
                                  unsigned int *status, cudaStream_t s)
{
    if (method == 0) {
        gdn_inv_fs_kernel<<<count, 128, 0, s>>>(A, T, C);
        return cudaGetLastError();
    }
    // 48 KB per CTA keeps at most four CTAs on an SM: four x 128 TMEM columns
    const int smem = 48 * 1024;
    cudaError_t e = cudaFuncSetAttribute(gdn_inv_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gdn_inv_tc_kernel<<<count, 128, smem, s>>>(A, T, C, status);
    return cudaGetLastError();
}
