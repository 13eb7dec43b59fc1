// Recurrent (token-by-token) gated delta rule for decoding, on CUDA cores.
//
// Per (sequence, head) and token, in the orientation S in R^{d_v x d_k}
// ("从零开始的 GDN 推导", recurrent form of the gated delta rule, with column
// vectors; "RNN的复兴03：现代RNN的并行计算", §一, the delta-rule update):
//
//     r   = S k                                 (what S retrieves for k)
//     S  <- alpha S + beta (v - alpha r) k^T    (= alpha S (I - beta k k^T) + beta v k^T)
//     o   = S q
//
// Every row of S evolves on its own: row i needs only S[i, :], k, q, v[i],
// alpha and beta.  A warp owns kRows rows of one (sequence, head) at a time,
// each row spread over the 32 lanes (four consecutive d_k elements per lane
// when d_k is a multiple of 4, else elements lane + 32 j), keeps them in
// registers across the call's tokens, and reduces the row dot products with
// one transposing butterfly for all kRows rows at once (9 shuffles instead of
// 5 per row).  The work is HBM-bound on the state: each step reads and writes
// d_v x d_k fp32 per (sequence, head); warps stride over (sequence, head, row
// group) items with a grid sized to fill every SM.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_internal.h"

namespace {

constexpr int kRows = 8;            // state rows per warp item
constexpr int kThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// The four elements of a d_k-long row that this lane owns (zeros past d_k).
template <bool VEC>
__device__ __forceinline__ void ld_row(const float *p, int dk, int lane, float (&x)[4])
{
    if (VEC) {
        if (4 * lane < dk) {
            const float4 u = *reinterpret_cast<const float4 *>(p + 4 * lane);
            x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
        } else {
            x[0] = x[1] = x[2] = x[3] = 0.f;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = lane + 32 * j < dk ? p[lane + 32 * j] : 0.f;
    }
}

template <bool VEC>
__device__ __forceinline__ void ld_row(const __nv_bfloat16 *p, int dk, int lane, float (&x)[4])
{
    if (VEC) {
        if (4 * lane < dk) {
            const uint2 u = *reinterpret_cast<const uint2 *>(p + 4 * lane);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
            x[0] = x[1] = x[2] = x[3] = 0.f;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = lane + 32 * j < dk ? to_f(p[lane + 32 * j]) : 0.f;
    }
}

template <bool VEC>
__device__ __forceinline__ void st_row(float *p, int dk, int lane, const float (&x)[4])
{
    if (VEC) {
        if (4 * lane < dk) *reinterpret_cast<float4 *>(p + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (lane + 32 * j < dk) p[lane + 32 * j] = x[j];
    }
}

// Sum of x[r] over the warp for each of the 8 values; lane l ends with the
// total of value (l >> 2) & 7.  Each halving step sends the half of its
// values that the partner keeps, so 4 + 2 + 1 shuffles reduce 8 values over
// lane groups of 8, and two more finish the sums over all 32 lanes.
__device__ __forceinline__ float reduce8(const float (&x)[kRows], int lane)
{
    float y[4], z[2];
    const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = u4 ? x[i] : x[i + 4];
        const float keep = u4 ? x[i + 4] : x[i];
        y[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = u3 ? y[i] : y[i + 2];
        const float keep = u3 ? y[i + 2] : y[i];
        z[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float w = (u2 ? z[1] : z[0]) + __shfl_xor_sync(0xffffffffu, u2 ? z[0] : z[1], 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    w += __shfl_xor_sync(0xffffffffu, w, 1);
    return w;
}

template <typename E, bool VEC>
__global__ void __launch_bounds__(kThreads) gdn_decode_kernel(const GdnDecodeArgs a)
{
    const int lane = threadIdx.x & 31;
    const long nwarps = (long)gridDim.x * (kThreads / 32);
    const int dk = a.dk, dv = a.dv, H = a.H, T = a.T;
    const int groups = (dv + kRows - 1) / kRows;
    const long items = (long)a.N * H * groups;
    const E *q = static_cast<const E *>(a.q), *k = static_cast<const E *>(a.k);
    const E *v = static_cast<const E *>(a.v);
    E *o = static_cast<E *>(a.o);
    const int my_row = (lane >> 2) & 7;  // the row whose sums this lane holds

    for (long it = (long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); it < items; it += nwarps) {
        const int g = (int)(it % groups);
        const long nh = it / groups;            // n * H + h
        const long n = nh / H;
        const int h = (int)(nh % H);
        const int r0 = g * kRows;
        const size_t sbase = (size_t)nh * dv * dk;

        float s[kRows][4];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (a.S_in && r0 + r < dv) {
                ld_row<VEC>(a.S_in + sbase + (size_t)(r0 + r) * dk, dk, lane, s[r]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) s[r][j] = 0.f;
            }
        }
        const bool row_ok = r0 + my_row < dv;

        for (int t = 0; t < T; ++t) {
            const size_t gi = ((size_t)n * T + t) * H + h;   // token-head index
            const float al = __expf(a.log_alpha[gi]);
            const float be = a.beta[gi];
            float kk[4], qq[4];
            ld_row<VEC>(k + gi * dk, dk, lane, kk);
            ld_row<VEC>(q + gi * dk, dk, lane, qq);
            const float vr = row_ok ? to_f(v[gi * dv + r0 + my_row]) : 0.f;

            // r = S k for the kRows rows; coefficient beta (v - alpha r) per row
            float d[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                d[r] = fmaf(s[r][0], kk[0], fmaf(s[r][1], kk[1], fmaf(s[r][2], kk[2], s[r][3] * kk[3])));
            const float rr = reduce8(d, lane);
            const float cf = be * (vr - al * rr);
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const float c = __shfl_sync(0xffffffffu, cf, 4 * r);
#pragma unroll
                for (int j = 0; j < 4; ++j) s[r][j] = fmaf(al, s[r][j], c * kk[j]);
            }
            // o = S q
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                d[r] = fmaf(s[r][0], qq[0], fmaf(s[r][1], qq[1], fmaf(s[r][2], qq[2], s[r][3] * qq[3])));
            const float oo = reduce8(d, lane);
            if ((lane & 3) == 0 && row_ok) from_f(o + gi * dv + r0 + my_row, oo);
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (r0 + r < dv) st_row<VEC>(a.S_out + sbase + (size_t)(r0 + r) * dk, dk, lane, s[r]);
    }
}

template <typename E, bool VEC>
cudaError_t launch(const GdnDecodeArgs &a, cudaStream_t s)
{
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gdn_decode_kernel<E, VEC>, kThreads, 0);
    if (e != cudaSuccess) return e;
    const long items = (long)a.N * a.H * ((a.dv + kRows - 1) / kRows);
    const long need = (items + kThreads / 32 - 1) / (kThreads / 32);
    long grid = (long)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > need) grid = need;
    gdn_decode_kernel<E, VEC><<<(unsigned)grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t gdn_launch_decode(const GdnDecodeArgs &a, cudaStream_t s, int *launches)
{
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool vec = a.dk % 4 == 0 && al16(a.q) && al16(a.k) && al16(a.S_out) &&
                     (a.S_in == nullptr || al16(a.S_in));
    cudaError_t e;
    if (a.dtype == 1)
        e = vec ? launch<__nv_bfloat16, true>(a, s) : launch<__nv_bfloat16, false>(a, s);
    else
        e = vec ? launch<float, true>(a, s) : launch<float, false>(a, s);
    *launches = e == cudaSuccess ? 1 : 0;
    return e;
}
