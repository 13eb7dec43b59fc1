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
// state are independent, so a CTA owns kRows rows of one (sequence, head) and
// the grid has dv / kRows x H x B CTAs.  Per step, M_s (d_k x d_k) sits in
// shared memory, each of the 8 warps multiplies the CTA's rows by its slice
// of d_k / 8 rows of M_s (a lane owns four columns, 16-byte accesses), and
// the eight partial products are summed with B_s into the next x.  The chain
// is short (one step per segment) and every step needs a whole M_s, which no
// step computes: all of them come from the propagator pass, so M_{s+1} and
// the CTA's rows of B_{s+1} are fetched by bulk copies (completing on an
// mbarrier) while step s computes, into the other of two buffers.  d_v is a
// multiple of 8 (the tensor-core path's rule), so a CTA's rows all exist.
#include <stdint.h>

#include "gdn_internal.h"

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kRows = 8;                       // state rows per CTA
constexpr uint64_t kScanWaitNs = 2000000000ull;  // bound on one copy's wait

__device__ __forceinline__ uint32_t su32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One bulk copy global -> this CTA's shared memory (16-byte aligned, size a
// multiple of 16), completing as tx bytes on `bar`.
// `expect` > 0: this copy also arrives on `bar` expecting that many bytes in
// all (the first copy of a step announces the step's total).
__device__ __forceinline__ void fetch(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                      uint32_t expect)
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of dst are done
    if (expect)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(expect)
                     : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool landed(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__global__ void __launch_bounds__(kScanThreads) gdn_scan_kernel(
    const float *__restrict__ S0, const float *__restrict__ Bseg, const float *__restrict__ Mseg,
    float *__restrict__ Sin, int P, int H, int dv, int dk, unsigned int *status)
{
    extern __shared__ __align__(16) float smem[];
    float *Ms = smem;                              // [2][dk][dk]
    float *Bs = Ms + 2 * dk * dk;                  // [2][kRows][dk]: this CTA's rows of B_s
    float *xT = Bs + 2 * kRows * dk;               // [dk][kRows]: the rows, transposed
    float *part = xT + dk * kRows;                 // [warps][kRows][dk] partial products
    uint64_t *bar = reinterpret_cast<uint64_t *>(part + kScanWarps * kRows * dk);  // [2]
    __shared__ int gave_up;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, b = blockIdx.z, r0 = blockIdx.x * kRows;
    const int kslice = dk / kScanWarps;            // d_k is a multiple of 8
    const bool lane_ok = 4 * lane < dk;
    const uint32_t mbytes = (uint32_t)(dk * dk * sizeof(float));
    const uint32_t bbytes = (uint32_t)(kRows * dk * sizeof(float));
    auto fetch_step = [&](int s) {  // M_s and this CTA's rows of B_s into buffer s & 1
        const size_t seg = (size_t)b * P + s;
        fetch(Ms + (s & 1) * dk * dk, Mseg + (seg * H + h) * dk * dk, mbytes, &bar[s & 1], mbytes + bbytes);
        fetch(Bs + (s & 1) * kRows * dk, Bseg + ((seg * H + h) * dv + r0) * dk, bbytes, &bar[s & 1], 0);
    };

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar[1])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        gave_up = 0;
    }
    for (int idx = tid; idx < kRows * dk; idx += kScanThreads) {
        const int r = idx / dk, i = idx % dk;
        xT[i * kRows + r] = S0 && r0 + r < dv ? S0[(((size_t)b * H + h) * dv + r0 + r) * dk + i] : 0.f;
    }
    __syncthreads();
    if (tid == 0 && P > 1) fetch_step(0);
    for (int s = 0; s < P; ++s) {
        const size_t row_base = (((size_t)b * P + s) * H + h) * dv + r0;
        for (int idx = tid; idx < kRows * dk; idx += kScanThreads) {
            const int r = idx / dk, i = idx % dk;
            if (r0 + r < dv) Sin[(row_base + r) * dk + i] = xT[i * kRows + r];
        }
        if (s == P - 1) break;
        // the other buffer was last read in step s - 1, which every thread has
        // left; one thread fetches and waits (bounded), the rest meet it below
        if (tid == 0) {
            if (s + 1 < P - 1 && !gave_up) fetch_step(s + 1);
            if (!gave_up && !landed(&bar[s & 1], (s >> 1) & 1)) {
                const uint64_t t0 = gtimer();
                while (!landed(&bar[s & 1], (s >> 1) & 1)) {
                    if (gtimer() - t0 > kScanWaitNs) {  // results invalid, flagged
                        gave_up = 1;
                        atomicOr(status, 0x2u);
                        break;
                    }
                }
            }
        }
        __syncthreads();
        const float *M = Ms + (s & 1) * dk * dk;
        float acc[kRows][4];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
        if (lane_ok) {
            for (int i = warp * kslice; i < (warp + 1) * kslice; ++i) {
                const float4 m = *reinterpret_cast<const float4 *>(M + i * dk + 4 * lane);
                const float4 x0 = *reinterpret_cast<const float4 *>(xT + i * kRows);
                const float4 x1 = *reinterpret_cast<const float4 *>(xT + i * kRows + 4);
                const float xr[kRows] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    acc[r][0] = fmaf(xr[r], m.x, acc[r][0]);
                    acc[r][1] = fmaf(xr[r], m.y, acc[r][1]);
                    acc[r][2] = fmaf(xr[r], m.z, acc[r][2]);
                    acc[r][3] = fmaf(xr[r], m.w, acc[r][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                *reinterpret_cast<float4 *>(part + (warp * kRows + r) * dk + 4 * lane) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        }
        __syncthreads();
        const float *Bv = Bs + (s & 1) * kRows * dk;
        for (int idx = tid; idx < kRows * dk; idx += kScanThreads) {
            const int r = idx / dk, c = idx % dk;
            float y = Bv[r * dk + c];
#pragma unroll
            for (int w = 0; w < kScanWarps; ++w) y += part[(w * kRows + r) * dk + c];
            xT[c * kRows + r] = y;
        }
        __syncthreads();
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
                            int B, int P, int H, int dv, int dk, unsigned int *status,
                            cudaStream_t s)
{
    const size_t smem = (2 * (size_t)dk * dk + (size_t)dk * kRows * (3 + kScanWarps)) * sizeof(float) +
                        2 * sizeof(uint64_t);
    cudaError_t e = cudaFuncSetAttribute(gdn_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((dv + kRows - 1) / kRows, H, B);
    gdn_scan_kernel<<<grid, kScanThreads, smem, s>>>(S0, Bseg, Mseg, Sin, P, H, dv, dk, status);
    return cudaGetLastError();
}

cudaError_t gdn_launch_segments(int32_t *cu, const int32_t *cu_seqlens, int B, int P, int T, int C,
                                unsigned int *status, cudaStream_t s)
{
    const int n = B * P + 1;
    gdn_segments_kernel<<<(n + 255) / 256, 256, 0, s>>>(cu, cu_seqlens, B, P, T, C, status);
    return cudaGetLastError();
}
