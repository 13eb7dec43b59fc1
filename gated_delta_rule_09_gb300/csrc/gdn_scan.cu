// Chunk-level scan over segments of long sequences, on CUDA cores (fp32).
//
// A sequence is cut into P segments at chunk boundaries.  The state after a
// segment is an affine function of the state before it,
//
//     S_end = S_start M_s + B_s,
//
// because every chunk step S <- e^{g_C} S + (U - W S^T)^T D K is affine in S
// ("从零开始的 GDN 推导", §"S 的推导"), and the composition of affine maps is
// associative ("Параллельность RNN?", §"Уровень 2: рекуррентность линейна, и
// потому ассоциативна", applied here to chunk operators instead of tokens).
// The propagator pass of the tcgen05 kernel produces
// M_s and B_s for every segment; this kernel chains them,
//
//     x_0 = S0,   x_{s+1} = x_s M_s + B_s,
//
// and writes every x_s, the state each segment starts from.  Rows of the
// state are independent: a warp owns two rows (four consecutive d_k elements
// per lane), M_s is staged once per step in shared memory for the CTA's 16
// rows, and x_s[i] is broadcast from the lane that holds it.
#include <stdint.h>

#include "gdn_internal.h"

namespace {

constexpr int kScanThreads = 256;
constexpr int kRowsPerCta = 16;  // 8 warps x 2 rows

__global__ void __launch_bounds__(kScanThreads) gdn_scan_kernel(
    const float *__restrict__ S0, const float *__restrict__ Bseg, const float *__restrict__ Mseg,
    float *__restrict__ Sin, int P, int H, int dv, int dk)
{
    extern __shared__ float Ms[];  // [dk][dk]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int r0 = blockIdx.x * kRowsPerCta + 2 * warp;
    const bool lane_ok = 4 * lane < dk;
    bool row_ok[2];
    float x[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        row_ok[r] = r0 + r < dv;
        const float *src = S0 && row_ok[r] && lane_ok
                               ? S0 + (((size_t)b * H + h) * dv + r0 + r) * dk + 4 * lane
                               : nullptr;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[r][e] = src ? src[e] : 0.f;
    }
    for (int s = 0; s < P; ++s) {
        const size_t seg = (size_t)b * P + s;
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (row_ok[r] && lane_ok) {
                float *dst = Sin + ((seg * H + h) * dv + r0 + r) * dk + 4 * lane;
                *reinterpret_cast<float4 *>(dst) = make_float4(x[r][0], x[r][1], x[r][2], x[r][3]);
            }
        if (s == P - 1) break;
        __syncthreads();  // every warp is done with the previous M_s
        const float4 *msrc = reinterpret_cast<const float4 *>(Mseg + (seg * H + h) * dk * dk);
        for (int i = threadIdx.x; i < dk * dk / 4; i += kScanThreads)
            reinterpret_cast<float4 *>(Ms)[i] = msrc[i];
        float y[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float *bsrc = row_ok[r] && lane_ok
                                    ? Bseg + ((seg * H + h) * dv + r0 + r) * dk + 4 * lane
                                    : nullptr;
#pragma unroll
            for (int e = 0; e < 4; ++e) y[r][e] = bsrc ? bsrc[e] : 0.f;
        }
        __syncthreads();
        for (int i4 = 0; i4 < dk / 4; ++i4) {
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const int i = 4 * i4 + e2;
                const float xa = __shfl_sync(0xffffffffu, x[0][e2], i4);
                const float xb = __shfl_sync(0xffffffffu, x[1][e2], i4);
                if (lane_ok) {
                    const float4 m = *reinterpret_cast<const float4 *>(Ms + i * dk + 4 * lane);
                    y[0][0] = fmaf(xa, m.x, y[0][0]); y[0][1] = fmaf(xa, m.y, y[0][1]);
                    y[0][2] = fmaf(xa, m.z, y[0][2]); y[0][3] = fmaf(xa, m.w, y[0][3]);
                    y[1][0] = fmaf(xb, m.x, y[1][0]); y[1][1] = fmaf(xb, m.y, y[1][1]);
                    y[1][2] = fmaf(xb, m.z, y[1][2]); y[1][3] = fmaf(xb, m.w, y[1][3]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[r][e] = y[r][e];
    }
}

// Segment boundaries as packed sequences: sequence b (tokens [s_b, e_b), from
// cu_seqlens when the input is packed, else [b T, (b + 1) T)) is cut into P
// segments of ceil(chunks_b / P) chunks each; trailing segments of a short
// sequence are empty.  Segment j of sequence b is unit b P + j, so the last
// segment of b ends where b + 1 starts.  A span that is negative or runs past
// T raises GDN_DEV_BAD_SEQLENS here and gets empty segments.
__global__ void gdn_segments_kernel(int32_t *cu, const int32_t *cu_seqlens, int B, int P, int T,
                                    int C, unsigned int *status)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int n = B * P;
    if (i > n) return;
    const int b = i / P, j = i % P;  // i == n: the end of the last sequence
    long s, e;
    if (cu_seqlens) {
        s = cu_seqlens[i == n ? B : b];
        e = i == n ? s : cu_seqlens[b + 1];
    } else {
        s = (long)(i == n ? B : b) * T;
        e = i == n ? s : s + T;
    }
    const long total = cu_seqlens ? (long)T : (long)B * T;
    if (s < 0 || e < s || e > total) {
        if (j == 0 || i == n) atomicOr(status, 0x1u);
        s = s < 0 ? 0 : (s > total ? total : s);
        e = s;
    }
    const long nch = (e - s + C - 1) / C, per = (nch + P - 1) / P;
    const long off = (long)j * per * C;
    cu[i] = (int32_t)(s + (off < e - s ? off : e - s));
}

}  // namespace

cudaError_t gdn_launch_scan(const float *S0, const float *Bseg, const float *Mseg, float *Sin,
                            int B, int P, int H, int dv, int dk, cudaStream_t s)
{
    const size_t smem = (size_t)dk * dk * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(gdn_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((dv + kRowsPerCta - 1) / kRowsPerCta, H, B);
    gdn_scan_kernel<<<grid, kScanThreads, smem, s>>>(S0, Bseg, Mseg, Sin, P, H, dv, dk);
    return cudaGetLastError();
}

cudaError_t gdn_launch_segments(int32_t *cu, const int32_t *cu_seqlens, int B, int P, int T, int C,
                                unsigned int *status, cudaStream_t s)
{
    const int n = B * P + 1;
    gdn_segments_kernel<<<(n + 255) / 256, 256, 0, s>>>(cu, cu_seqlens, B, P, T, C, status);
    return cudaGetLastError();
}
