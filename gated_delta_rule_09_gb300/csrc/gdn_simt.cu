// fp32 CUDA-core kernel for the chunkwise gated delta rule forward pass.
//
// One CTA owns one (sequence, head, 32-wide d_v tile) and walks that
// sequence's chunks in order, holding its slice of the state S (d_v x d_k,
// fp32) in shared memory.  Per chunk of n <= C tokens it takes the steps of
// "从零开始的 GDN 推导" §"总结" in the column-vector orientation:
//
//   g      inclusive cumulative sum of log(alpha) inside the chunk
//   A      StrictLower(diag(beta) K K^T * e^{g_i - g_j})        (§"UT transform")
//   T      (I + A)^{-1} by column-wise forward substitution
//          ("RNN的复兴03：现代RNN的并行计算", §2.3.1, with the sign of A flipped)
//   W, U   T diag(beta) (K * e^g),  T diag(eta) V                (§"S 的推导";
//          eta, the write strength, is beta unless given)
//   V_new  U - W S^T
//   O      (Q * e^g) S^T + (Q K^T * e^{g_i - g_j}, j <= i) V_new (§"O 的推导")
//   S      e^{g_last} S + V_new^T (K * e^{g_last - g})          (§"S 的推导")
//
// All arithmetic is fp32; inputs are widened on load (fp32 or bf16) and the
// output is rounded once to the input dtype.  This kernel serves the fp32
// dtype (where bf16 tensor-core operands would miss a 1e-4 relative error
// budget) and every shape the tcgen05 kernel does not cover.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kDvt = 32;  // d_v columns per CTA

__device__ __forceinline__ float ld_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_out(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads)
gdn_simt_kernel(GdnArgs a)
{
    const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x;
    const int C = a.C, dk = a.dk, H = a.H, dv = a.dv;
    const int v0 = tile * kDvt;
    const int nv = min(kDvt, dv - v0);
    const TIn *q = static_cast<const TIn *>(a.q);
    const TIn *k = static_cast<const TIn *>(a.k);
    const TIn *v = static_cast<const TIn *>(a.v);
    TIn *o = static_cast<TIn *>(a.o);

    long start, len;
    if (a.cu_seqlens) {
        const int s = a.cu_seqlens[n], e = a.cu_seqlens[n + 1];
        if (s < 0 || e < s || e > a.T) {
            if (tid == 0) atomicOr(a.status, 1u);
            return;
        }
        start = s;
        len = e - s;
    } else {
        start = (long)n * a.T;
        len = a.T;
    }

    extern __shared__ float sm[];
    const int ldk = dk + 1, ldc = C + 1, ldv = kDvt + 1;
    float *Ks = sm;                 // [C][ldk]
    float *Qs = Ks + C * ldk;       // [C][ldk]
    float *Ws = Qs + C * ldk;       // [C][ldk]
    float *Ss = Ws + C * ldk;       // [kDvt][ldk]  state slice S[v0 + r][:]
    float *As = Ss + kDvt * ldk;    // [C][ldc]
    float *Ts = As + C * ldc;       // [C][ldc]
    float *Ps = Ts + C * ldc;       // [C][ldc]
    float *Vs = Ps + C * ldc;       // [C][ldv]
    float *Us = Vs + C * ldv;       // [C][ldv]  U, then V_new
    float *g = Us + C * ldv;        // [C]
    float *eg = g + C;              // [C]  e^{g_i}
    float *ek = eg + C;             // [C]  e^{g_last - g_i}
    float *bt = ek + C;             // [C]  beta
    float *et = bt + C;             // [C]  eta (the write strength; beta unless given)

    const size_t sbase = ((size_t)n * H + h) * dv * dk;
    for (int idx = tid; idx < kDvt * dk; idx += kThreads) {
        const int r = idx / dk, c = idx % dk;
        float x = 0.f;
        if (a.S0 && r < nv) x = a.S0[sbase + (size_t)(v0 + r) * dk + c];
        Ss[r * ldk + c] = x;
    }

    for (long c0 = 0; c0 < len; c0 += C) {
        const int nc = (int)min((long)C, len - c0);
        __syncthreads();
        for (int idx = tid; idx < C * dk; idx += kThreads) {
            const int i = idx / dk, c = idx % dk;
            float kx = 0.f, qx = 0.f;
            if (i < nc) {
                const size_t off = ((size_t)(start + c0 + i) * H + h) * dk + c;
                kx = ld_in(k, off);
                qx = ld_in(q, off);
            }
            Ks[i * ldk + c] = kx;
            Qs[i * ldk + c] = qx;
        }
        for (int idx = tid; idx < C * kDvt; idx += kThreads) {
            const int i = idx / kDvt, r = idx % kDvt;
            float x = 0.f;
            if (i < nc && r < nv) x = ld_in(v, ((size_t)(start + c0 + i) * H + h) * dv + v0 + r);
            Vs[i * ldv + r] = x;
        }
        if (tid < C) {
            float la = 0.f, b = 0.f, e = 0.f;
            if (tid < nc) {
                const size_t gi = (size_t)(start + c0 + tid) * H + h;
                la = a.log_alpha[gi];
                b = a.beta[gi];
                e = a.eta ? a.eta[gi] : b;
            }
            g[tid] = la;
            bt[tid] = b;
            et[tid] = e;
        }
        __syncthreads();
        if (tid == 0) {  // inclusive cumulative sum (padding rows add 0)
            float acc = 0.f;
            for (int i = 0; i < C; ++i) {
                acc += g[i];
                g[i] = acc;
            }
        }
        __syncthreads();
        const float glast = g[C - 1];
        if (tid < C) {
            eg[tid] = expf(g[tid]);
            ek[tid] = expf(glast - g[tid]);
        }
        // A (strictly lower) and P = (Q K^T) * decay (lower, diagonal kept)
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int i = idx / C, j = idx % C;
            float kk = 0.f, qk = 0.f, d = 0.f;
            if (j <= i) {
                const float *ki = Ks + i * ldk, *kj = Ks + j * ldk, *qi = Qs + i * ldk;
                for (int c = 0; c < dk; ++c) {
                    kk = fmaf(ki[c], kj[c], kk);
                    qk = fmaf(qi[c], kj[c], qk);
                }
                d = expf(g[i] - g[j]);
            }
            As[i * ldc + j] = (j < i) ? bt[i] * kk * d : 0.f;
            Ps[i * ldc + j] = (j <= i) ? qk * d : 0.f;
        }
        __syncthreads();
        // T = (I + A)^{-1}: thread j owns column j; rows in order.
        if (tid < C) {
            const int j = tid;
            for (int i = 0; i < C; ++i) Ts[i * ldc + j] = (i == j) ? 1.f : 0.f;
            for (int i = j + 1; i < C; ++i) {
                float acc = 0.f;
                for (int m = j; m < i; ++m) acc = fmaf(As[i * ldc + m], Ts[m * ldc + j], acc);
                Ts[i * ldc + j] = -acc;
            }
        }
        __syncthreads();
        // W = T diag(beta) (K * e^g),  U = T diag(eta) V
        for (int idx = tid; idx < C * dk; idx += kThreads) {
            const int i = idx / dk, c = idx % dk;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j)
                acc = fmaf(Ts[i * ldc + j], bt[j] * eg[j] * Ks[j * ldk + c], acc);
            Ws[i * ldk + c] = acc;
        }
        for (int idx = tid; idx < C * kDvt; idx += kThreads) {
            const int i = idx / kDvt, r = idx % kDvt;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j)
                acc = fmaf(Ts[i * ldc + j], et[j] * Vs[j * ldv + r], acc);
            Us[i * ldv + r] = acc;
        }
        __syncthreads();
        // V_new = U - W S^T
        for (int idx = tid; idx < C * kDvt; idx += kThreads) {
            const int i = idx / kDvt, r = idx % kDvt;
            const float *wi = Ws + i * ldk, *sr = Ss + r * ldk;
            float acc = 0.f;
            for (int c = 0; c < dk; ++c) acc = fmaf(wi[c], sr[c], acc);
            Us[i * ldv + r] -= acc;
        }
        __syncthreads();
        // O = e^{g_i} (Q S^T)_i + sum_{j <= i} P_ij V_new_j
        for (int idx = tid; idx < C * kDvt; idx += kThreads) {
            const int i = idx / kDvt, r = idx % kDvt;
            if (i < nc && r < nv) {
                const float *qi = Qs + i * ldk, *sr = Ss + r * ldk;
                float acc = 0.f;
                for (int c = 0; c < dk; ++c) acc = fmaf(qi[c], sr[c], acc);
                acc *= eg[i];
                for (int j = 0; j <= i; ++j) acc = fmaf(Ps[i * ldc + j], Us[j * ldv + r], acc);
                st_out(o, ((size_t)(start + c0 + i) * H + h) * dv + v0 + r, acc);
            }
        }
        __syncthreads();
        // S = e^{g_last} S + V_new^T (K * e^{g_last - g})
        const float dl = expf(glast);
        for (int idx = tid; idx < kDvt * dk; idx += kThreads) {
            const int r = idx / dk, c = idx % dk;
            float acc = 0.f;
            for (int j = 0; j < nc; ++j)
                acc = fmaf(Us[j * ldv + r], Ks[j * ldk + c] * ek[j], acc);
            Ss[r * ldk + c] = fmaf(dl, Ss[r * ldk + c], acc);
        }
    }
    __syncthreads();
    if (a.S_final) {
        for (int idx = tid; idx < kDvt * dk; idx += kThreads) {
            const int r = idx / dk, c = idx % dk;
            if (r < nv) a.S_final[sbase + (size_t)(v0 + r) * dk + c] = Ss[r * ldk + c];
        }
    }
}

}  // namespace

size_t gdn_simt_smem_bytes(int C, int dk)
{
    const size_t ldk = dk + 1, ldc = C + 1, ldv = kDvt + 1;
    return sizeof(float) * (3 * C * ldk + kDvt * ldk + 3 * C * ldc + 2 * C * ldv + 5 * C);
}

cudaError_t gdn_launch_simt(const GdnArgs &a, cudaStream_t s, int *launches)
{
    const size_t smem = gdn_simt_smem_bytes(a.C, a.dk);
    dim3 grid((a.dv + kDvt - 1) / kDvt, a.H, a.N);
    cudaError_t e;
    if (a.dtype == 1) {
        e = cudaFuncSetAttribute(gdn_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        gdn_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
    } else {
        e = cudaFuncSetAttribute(gdn_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        gdn_simt_kernel<float><<<grid, kThreads, smem, s>>>(a);
    }
    *launches = 1;
    return cudaGetLastError();
}
