// Internal interface between the C-ABI front end (gdn_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

struct GdnArgs {
    const void *q, *k, *v;       // [*, T, H, dk] / [*, T, H, dv], dtype
    const float *log_alpha;      // [*, T, H]
    const float *beta;           // [*, T, H]
    const float *eta;            // [*, T, H] write strength, or null (= beta)
    const float *S0;             // [N, H, dv, dk] or null
    void *o;                     // [*, T, H, dv], dtype
    float *S_final;              // [N, H, dv, dk] or null
    int N, H, T, dk, dv, C;
    const int32_t *cu_seqlens;   // device [N + 1] or null
    int dtype;                   // 0 = fp32, 1 = bf16
    unsigned int *status;        // device status word (GDN_DEV_* bits)
    // 0: the forward pass.  1: segment propagators for the chunk-level scan
    // (tcgen05 kernel only): per sequence, the state reached from zero (into
    // S_final) and the d_k x d_k transition M of S_end = S_start M + that
    // state (into prop_M, [N, H, dk, dk]); no outputs are written.
    int mode;
    float *prop_M;
};

// fp32 CUDA-core kernel: every supported shape and dtype.
cudaError_t gdn_launch_simt(const GdnArgs &a, cudaStream_t s, int *launches);
size_t gdn_simt_smem_bytes(int C, int dk);

// tcgen05 tensor-core kernel: bf16, the shapes gdn_tc_supported() accepts.
bool gdn_tc_supported(const GdnArgs &a);
cudaError_t gdn_launch_tc(const GdnArgs &a, cudaStream_t s, int *launches);

struct GdnDecodeArgs {
    const void *q, *k, *v;       // [N, T, H, dk] / [N, T, H, dv], dtype
    const float *log_alpha;      // [N, T, H]
    const float *beta;           // [N, T, H]
    const float *S_in;           // [N, H, dv, dk] or null (zeros)
    void *o;                     // [N, T, H, dv], dtype
    float *S_out;                // [N, H, dv, dk]; may equal S_in
    int N, H, T, dk, dv;
    int dtype;                   // 0 = fp32, 1 = bf16
};

// Recurrent (token-by-token) kernel for decoding, on CUDA cores.
cudaError_t gdn_launch_decode(const GdnDecodeArgs &a, cudaStream_t s, int *launches);

// Chunk-level scan over segments: x_{s+1} = x_s M_s + B_s (fp32, CUDA cores).
cudaError_t gdn_launch_scan(const float *S0, const float *Bseg, const float *Mseg, float *Sin,
                            int B, int P, int H, int dv, int dk, unsigned int *status,
                            cudaStream_t s);
// Segment boundaries: sequence b (B sequences of T tokens, or packed through
// cu_seqlens) cut into P segments of ceil(chunks_b / P) chunks each.
cudaError_t gdn_launch_segments(int32_t *cu, const int32_t *cu_seqlens, int B, int P, int T, int C,
                                unsigned int *status, cudaStream_t s);

// Batched UT inverse T = (I + StrictLower(A))^{-1}, C <= 64: method 0 blocked
// forward substitution (CUDA cores, fp32), 1 doubling product (tcgen05).
cudaError_t gdn_launch_ut_inverse(const float *A, float *T, int count, int C, int method,
                                  unsigned int *status, cudaStream_t s);
