// tcgen05 tensor-core kernel for the chunkwise gated delta rule (bf16 in/out,
// fp32 state and accumulation, fp16 tensor-core operands) on sm_103a.
//
// One CTA (4 warps) owns one (sequence, head, 128-wide d_v tile) and walks the
// sequence's chunks of C = 64 tokens in order.  The d_v x d_k state slice lives
// in TMEM as an fp32 MMA accumulator for the whole walk.  Per chunk, in the
// notation of "从零开始的 GDN 推导" (§"UT transform", §"S 的推导", §"O 的推导",
// §"总结") transposed so that S is d_v x d_k (g = in-chunk cumulative log-decay):
//
//   batch 1  [K;Q] K^T -> K K^T, Q K^T           S Q^T                (tcgen05)
//   A   = StrictLower(diag(beta) K K^T * e^{g_i-g_j})                 (CUDA cores)
//   P   = Lower(Q K^T * e^{g_i-g_j})                                  (CUDA cores)
//   T   = (I + A)^{-1}, blocked forward substitution in shared memory  (CUDA cores)
//   batch 2  W^T = K^T (T diag(beta e^g))^T,  U^T = V^T (T diag(beta))^T
//   batch 3  S W^T
//   V_new^T = U^T - S W^T   (fp16 copy, and a copy scaled by e^{g_C - g_j})
//   batch 4  O^T_intra = V_new^T P^T,   S <- e^{g_C} S + (V_new * e^{g_C-g})^T K
//   o_i = e^{g_i} (S Q^T)_i + O_intra_i  -> bf16
//
// Every MMA has M = 128 (d_k or the d_v tile on the M side), so each row of a
// result is one TMEM lane and one thread of the epilogue owns it.  Operands
// are fp16 (11-bit significand): the bf16 q/k/v tiles are converted in shared
// memory after they land (exact for |x| < 65504) and every operand written by
// the epilogues is fp16; accumulation and the state stay fp32.  bf16 operands
// throughout would leave about 0.03 x RMS of error in o on these workloads, fp16
// about 0.003.  A value outside the fp16 range raises GDN_DEV_F16_RANGE.  Operands
// are 128-byte-swizzled shared-memory tiles; q/k/v tiles arrive by TMA (the
// next chunk's q/k while the current one computes), the rest are written by
// the epilogue threads.  Every mbarrier wait is bounded: on timeout the CTA
// sets GDN_DEV_WAIT_TIMEOUT, drains its own TMA copies, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <mutex>

#include "gdn_internal.h"
#include "sm100_ptx.cuh"

namespace {

using namespace sm100;

constexpr int kC = 64;       // chunk length
constexpr int kDK = 128;     // d_k
constexpr int kDVT = 128;    // d_v columns per CTA
constexpr int kThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// shared-memory plan (bytes from a 1024-aligned base)
constexpr int kKQStage = 32768;                 // 2 d_k-halves x [K rows 0-63 | Q rows 64-127] x 128 B
constexpr int kOffKQ = 0;                       // 2 stages
constexpr int kOffV = kOffKQ + 2 * kKQStage;    // 2 d_v-halves x 64 rows x 128 B
constexpr int kOffSb = kOffV + 16384;           // S (fp16), 2 d_k-halves x 128 rows x 128 B
constexpr int kOffR = kOffSb + 32768;           // Ws | VnT | VnTs  (aliased by A, T, X fp32)
constexpr int kOffWs = kOffR;
constexpr int kOffVnT = kOffR + 16384;
constexpr int kOffVnTs = kOffR + 32768;
constexpr int kOffPm = kOffR + 49152;
constexpr int kOffTpp = kOffPm + 8192;
constexpr int kOffTp = kOffTpp + 8192;
constexpr int kOffSmall = kOffTp + 8192;
constexpr int kLdA = 65;                        // padded fp32 row stride of A / T
constexpr int kSmemBytes = kOffSmall + 2048 + 1024;  // + small arrays + alignment slack

// tensor-memory columns
constexpr uint32_t kColKQ = 0, kColSQ = 64, kColW = 128, kColU = 192, kColSW = 256,
                   kColO = 320, kColS = 384;

struct Small {
    float g[kC], eg[kC], ekc[kC], beta[kC], scan[kC];
    uint64_t bar_kq[2], bar_v, bar_mma;
    uint32_t tmem;
    int abort_flag;
};
static_assert(sizeof(Small) <= 2048, "small shared block");

constexpr float kF16Max = 65504.f;

__device__ __forceinline__ uint32_t pack_f16(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Write 8 consecutive values of row r, 16-byte chunk c, of a swizzled tile as
// fp16, folding their magnitudes into *amax for the range check.
__device__ __forceinline__ void st_chunk(uint8_t *tile, int r, int c, const float *x, float *amax)
{
    uint4 u;
    u.x = pack_f16(x[0], x[1]);
    u.y = pack_f16(x[2], x[3]);
    u.z = pack_f16(x[4], x[5]);
    u.w = pack_f16(x[6], x[7]);
    float m = *amax;
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(x[e]));
    *amax = m;
    *reinterpret_cast<uint4 *>(tile + sw128(r, c)) = u;
}

// bf16 -> fp16 for the 8 values of one 16-byte chunk, in place.
__device__ __forceinline__ void chunk_bf16_to_f16(uint8_t *p, float *amax)
{
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float m = *amax;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
        w[e] = pack_f16(f.x, f.y);
    }
    *amax = m;
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t lane_addr(uint32_t tbase, int warp, uint32_t col)
{
    return tbase + (static_cast<uint32_t>(warp * 32) << 16) + col;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, Small *s,
                                              unsigned int *status)
{
    if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
    s->abort_flag = 1;
    atomicOr(status, 0x2u);
    return false;
}

__global__ void __launch_bounds__(kThreads, 1)
gdn_tc_kernel(const GdnArgs a, const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Small *s = reinterpret_cast<Small *>(sm + kOffSmall);
    float *As = reinterpret_cast<float *>(sm + kOffR);            // [64][65]
    float *Ts = As + kC * kLdA;                                    // [64][65]
    float *Xs = Ts + kC * kLdA;                                    // [32][33]
    uint8_t *Sb = sm + kOffSb, *Vt = sm + kOffV, *Ws = sm + kOffWs, *VnT = sm + kOffVnT,
            *VnTs = sm + kOffVnTs, *Pm = sm + kOffPm, *Tpp = sm + kOffTpp, *Tp = sm + kOffTp;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vt = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = a.H, dv = a.dv;
    const int v0 = vt * kDVT;

    long start = 0, len = 0;
    bool bad = false;
    if (a.cu_seqlens) {
        const int s0 = a.cu_seqlens[n], e0 = a.cu_seqlens[n + 1];
        if (s0 < 0 || e0 < s0 || e0 > a.T) bad = true;
        else { start = s0; len = e0 - s0; }
    } else {
        start = (long)n * a.T;
        len = a.T;
    }
    if (bad) {  // uniform across the CTA: nothing allocated yet
        if (tid == 0) atomicOr(a.status, 0x1u);
        return;
    }
    const int nchunks = (int)((len + kC - 1) / kC);

    if (warp == 0) {
        tmem_alloc(&s->tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&s->bar_kq[0], 1);
        mbar_init(&s->bar_kq[1], 1);
        mbar_init(&s->bar_v, 1);
        mbar_init(&s->bar_mma, 1);
        s->abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s->tmem;

    // q/k tiles of chunk c into stage (c & 1); v tile into the single V buffer
    auto issue_kq = [&](int c) {
        uint8_t *kq = sm + kOffKQ + (c & 1) * kKQStage;
        const int z = (int)(start + (long)c * kC);
        mbar_arrive_expect_tx(&s->bar_kq[c & 1], 4 * 8192);
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(kq + b * 16384, &tm_k, &s->bar_kq[c & 1], b * 64, h, z);
            tma_load_3d(kq + b * 16384 + 8192, &tm_q, &s->bar_kq[c & 1], b * 64, h, z);
        }
    };
    auto issue_v = [&](int c) {
        const int z = (int)(start + (long)c * kC);
        mbar_arrive_expect_tx(&s->bar_v, 2 * 8192);
        for (int b = 0; b < 2; ++b)
            tma_load_3d(Vt + b * 8192, &tm_v, &s->bar_v, v0 + b * 64, h, z);
    };
    // outstanding-copy bookkeeping (thread 0 only) for draining on abort
    int kq_issued = 0, v_issued = 0;
    if (tid == 0 && nchunks > 0) {
        issue_kq(0);
        issue_v(0);
        kq_issued = 1;
        v_issued = 1;
    }

    // initial state into the TMEM accumulator (lane = d_v row)
    {
        const float *src = a.S0 ? a.S0 + (((size_t)n * H + h) * dv + v0 + tid) * kDK : nullptr;
        for (int cb = 0; cb < 4; ++cb) {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = src ? src[cb * 32 + j] : 0.f;
            tmem_st32(lane_addr(tbase, warp, kColS + cb * 32), x);
        }
        tmem_st_wait();
    }

    // gates of the next chunk, prefetched into registers by threads 0..63
    float la_next = 0.f, b_next = 0.f;
    auto load_gates = [&](int c) {
        la_next = 0.f;
        b_next = 0.f;
        if (tid < kC && c < nchunks) {
            const long t = (long)c * kC + tid;
            if (t < len) {
                const size_t gi = (size_t)(start + t) * H + h;
                la_next = a.log_alpha[gi];
                b_next = a.beta[gi];
            }
        }
    };
    load_gates(0);

    uint32_t mma_phase = 0;
    float amax = 0.f;  // largest magnitude this thread converted to fp16
    int c = 0;
    for (; c < nchunks; ++c) {
        const int nc = (int)min((long)kC, len - (long)c * kC);
        const long tok0 = start + (long)c * kC;
        uint8_t *kq = sm + kOffKQ + (c & 1) * kKQStage;

        // -------- decay: g = inclusive cumulative sum of log alpha (padding adds 0)
        const float la = la_next, bt = b_next;
        load_gates(c + 1);
        if (tid < kC) {
            float x = la;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            s->scan[tid] = x;
            s->beta[tid] = bt;
        }
        __syncthreads();
        if (tid < kC) s->g[tid] = s->scan[tid] + (tid >= 32 ? s->scan[31] : 0.f);
        __syncthreads();
        const float gC = s->g[kC - 1];
        if (tid < kC) {
            s->eg[tid] = __expf(s->g[tid]);
            s->ekc[tid] = __expf(gC - s->g[tid]);
        }
        // next chunk's q/k into the other stage (free since the previous chunk ended)
        if (tid == 0 && c + 1 < nchunks) {
            issue_kq(c + 1);
            ++kq_issued;
        }

        // -------- this chunk's tiles
        if (!wait_or_abort(&s->bar_kq[c & 1], (c >> 1) & 1, s, a.status)) {}
        if (!wait_or_abort(&s->bar_v, c & 1, s, a.status)) {}
        // bf16 -> fp16 in place; rows past the sequence are zeroed (they may
        // hold another sequence).  Six 64-row tiles: K, Q for both d_k halves,
        // V for both d_v halves; 8 chunks of 16 B per row.
        for (int idx = tid; idx < 6 * kC * 8; idx += kThreads) {
            const int tile = idx / (kC * 8), r = (idx / 8) % kC, cc = idx % 8;
            uint8_t *base = tile < 4 ? kq + (tile >> 1) * 16384 + (tile & 1) * 8192
                                     : Vt + (tile - 4) * 8192;
            uint8_t *p = base + sw128(r, cc);
            if (r < nc) chunk_bf16_to_f16(p, &amax);
            else *reinterpret_cast<uint4 *>(p) = make_uint4(0, 0, 0, 0);
        }

        // -------- incoming state: fp16 copy for the MMAs, TMEM <- e^{g_C} S
        {
            const float dC = __expf(gC);
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(lane_addr(tbase, warp, kColS + cb * 32), x);
                tmem_ld_wait();
                uint8_t *box = Sb + (cb >> 1) * 16384;
#pragma unroll
                for (int q = 0; q < 4; ++q) st_chunk(box, tid, (cb & 1) * 4 + q, x + q * 8, &amax);
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] *= dC;
                tmem_st32(lane_addr(tbase, warp, kColS + cb * 32), x);
            }
            tmem_st_wait();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (s->abort_flag) break;

        // -------- batch 1: [K;Q] K^T  and  S Q^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_f16_f32(128, 64, 0, 0);
            const uint32_t kqa = smem_u32(kq), sba = smem_u32(Sb);
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_f16kind(tbase + kColKQ, sdesc_sw128(kqa + o, 16, 1024),
                         sdesc_sw128(kqa + o, 16, 1024), id, ks > 0);
                mma_f16kind(tbase + kColSQ, sdesc_sw128(sba + o, 16, 1024),
                         sdesc_sw128(kqa + o + 8192, 16, 1024), id, ks > 0);
            }
            mma_commit(&s->bar_mma);
        }
        wait_or_abort(&s->bar_mma, mma_phase, s, a.status);
        mma_phase ^= 1;
        tc_fence_after();

        // -------- A (fp32, rows 0-63) and P (fp16, rows 64-127)
        {
            const bool is_k = tid < kC;
            const int i = is_k ? tid : tid - kC;
            const float gi = s->g[i];
            const float bi = s->beta[i];
            float x[32];
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(lane_addr(tbase, warp, kColKQ + half * 32), x);
                tmem_ld_wait();
                if (is_k) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int j = half * 32 + jj;
                        As[i * kLdA + j] = (j < i) ? bi * x[jj] * __expf(gi - s->g[j]) : 0.f;
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int j = half * 32 + jj;
                        x[jj] = (j <= i) ? x[jj] * __expf(gi - s->g[j]) : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) st_chunk(Pm, i, half * 4 + q, x + q * 8, &amax);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // -------- T = (I + A)^{-1}
        // (1) the four 16x16 diagonal blocks, one warp each: lane l < 16 owns
        //     column l of its block and substitutes forward down the rows.
        {
            const int b = warp, l = lane;
            float t[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) t[r] = (r == l) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m)
                    if (m >= l) acc = fmaf(As[(16 * b + r) * kLdA + 16 * b + m], t[m], acc);
                if (r > l) t[r] = -acc;
            }
            if (l < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) Ts[(16 * b + r) * kLdA + 16 * b + l] = t[r];
            }
        }
        __syncthreads();
        // (2) 16 -> 32: T[1,0] = -T11 (A10 T00) for the block pairs (0,1), (2,3)
        for (int idx = tid; idx < 512; idx += kThreads) {
            const int p = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            const int R = 16 * (2 * p + 1), Cc = 32 * p;
            float acc = 0.f;
            for (int m = cc; m < 16; ++m)
                acc = fmaf(As[(R + r) * kLdA + Cc + m], Ts[(Cc + m) * kLdA + Cc + cc], acc);
            Xs[p * 16 * 17 + r * 17 + cc] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < 512; idx += kThreads) {
            const int p = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
            const int R = 16 * (2 * p + 1), Cc = 32 * p;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc = fmaf(Ts[(R + r) * kLdA + R + m], Xs[p * 16 * 17 + m * 17 + cc], acc);
            Ts[(R + r) * kLdA + Cc + cc] = -acc;
        }
        __syncthreads();
        // (3) 32 -> 64: T[32:64, 0:32] = -T2 (A21 T1)
        for (int idx = tid; idx < 1024; idx += kThreads) {
            const int r = idx >> 5, cc = idx & 31;
            float acc = 0.f;
            for (int m = cc; m < 32; ++m)
                acc = fmaf(As[(32 + r) * kLdA + m], Ts[m * kLdA + cc], acc);
            Xs[r * 33 + cc] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < 1024; idx += kThreads) {
            const int r = idx >> 5, cc = idx & 31;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m)
                acc = fmaf(Ts[(32 + r) * kLdA + 32 + m], Xs[m * 33 + cc], acc);
            Ts[(32 + r) * kLdA + cc] = -acc;
        }
        __syncthreads();
        // T'' = T diag(beta e^g) (rows 0-63 by threads 0-63), T' = T diag(beta) (threads 64-127)
        {
            const bool first = tid < kC;
            const int j = first ? tid : tid - kC;
            uint8_t *dst = first ? Tpp : Tp;
            float x[8];
            for (int q = 0; q < 8; ++q) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int cc = q * 8 + e;
                    const float sc = first ? s->beta[cc] * s->eg[cc] : s->beta[cc];
                    x[e] = (cc <= j) ? Ts[j * kLdA + cc] * sc : 0.f;
                }
                st_chunk(dst, j, q, x, &amax);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // -------- batch 2: W^T = K^T T''^T (A: K as MN-major),  U^T = V^T T'^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idw = idesc_f16_f32(128, 64, 1, 0);
            const uint32_t kqa = smem_u32(kq), va = smem_u32(Vt);
            for (int ks = 0; ks < 4; ++ks) {
                mma_f16kind(tbase + kColW, sdesc_sw128(kqa + ks * 2048, 16384, 1024),
                         sdesc_sw128(smem_u32(Tpp) + ks * 32, 16, 1024), idw, ks > 0);
                mma_f16kind(tbase + kColU, sdesc_sw128(va + ks * 2048, 8192, 1024),
                         sdesc_sw128(smem_u32(Tp) + ks * 32, 16, 1024), idw, ks > 0);
            }
            mma_commit(&s->bar_mma);
        }
        wait_or_abort(&s->bar_mma, mma_phase, s, a.status);
        mma_phase ^= 1;
        tc_fence_after();
        // V buffer is free: fetch the next chunk's values
        if (tid == 0 && c + 1 < nchunks) {
            issue_v(c + 1);
            ++v_issued;
        }

        // -------- W^T rows (lane = d) -> Ws as the MN-major B operand of S W^T
        {
            float x[32];
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(lane_addr(tbase, warp, kColW + half * 32), x);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) st_chunk(Ws, tid, half * 4 + q, x + q * 8, &amax);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // -------- batch 3: S W^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_f16_f32(128, 64, 0, 1);
            const uint32_t sba = smem_u32(Sb), wsa = smem_u32(Ws);
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_f16kind(tbase + kColSW, sdesc_sw128(sba + o, 16, 1024),
                         sdesc_sw128(wsa + ks * 2048, 8192, 1024), id, ks > 0);
            }
            mma_commit(&s->bar_mma);
        }
        wait_or_abort(&s->bar_mma, mma_phase, s, a.status);
        mma_phase ^= 1;
        tc_fence_after();

        // -------- V_new^T = U^T - S W^T  (row v = tid)
        {
            float u[32], w[32];
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(lane_addr(tbase, warp, kColU + half * 32), u);
                tmem_ld32(lane_addr(tbase, warp, kColSW + half * 32), w);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) u[j] -= w[j];
#pragma unroll
                for (int q = 0; q < 4; ++q) st_chunk(VnT, tid, half * 4 + q, u + q * 8, &amax);
#pragma unroll
                for (int j = 0; j < 32; ++j) u[j] *= s->ekc[half * 32 + j];
#pragma unroll
                for (int q = 0; q < 4; ++q) st_chunk(VnTs, tid, half * 4 + q, u + q * 8, &amax);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // -------- batch 4: O_intra^T = V_new^T P^T;  S += (V_new e^{gC-g})^T K
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ido = idesc_f16_f32(128, 64, 0, 0);
            const uint32_t ids = idesc_f16_f32(128, 128, 0, 1);
            const uint32_t kqa = smem_u32(kq);
            for (int ks = 0; ks < 4; ++ks) {
                mma_f16kind(tbase + kColO, sdesc_sw128(smem_u32(VnT) + ks * 32, 16, 1024),
                         sdesc_sw128(smem_u32(Pm) + ks * 32, 16, 1024), ido, ks > 0);
                mma_f16kind(tbase + kColS, sdesc_sw128(smem_u32(VnTs) + ks * 32, 16, 1024),
                         sdesc_sw128(kqa + ks * 2048, 16384, 1024), ids, 1);
            }
            mma_commit(&s->bar_mma);
        }
        wait_or_abort(&s->bar_mma, mma_phase, s, a.status);
        mma_phase ^= 1;
        tc_fence_after();

        // -------- o_i = e^{g_i} (S Q^T)[v][i] + O_intra^T[v][i]
        {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o);
            const size_t col = (size_t)v0 + tid;
            float x[32], y[32];
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(lane_addr(tbase, warp, kColSQ + half * 32), x);
                tmem_ld32(lane_addr(tbase, warp, kColO + half * 32), y);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int i = half * 32 + j;
                    if (i < nc)
                        o[((size_t)(tok0 + i) * H + h) * dv + col] =
                            __float2bfloat16_rn(fmaf(s->eg[i], x[j], y[j]));
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (s->abort_flag) break;
    }

    if (amax > kF16Max) atomicOr(a.status, 0x4u);

    // -------- final state, or drain after an abort
    if (!s->abort_flag) {
        if (a.S_final) {
            float *dst = a.S_final + (((size_t)n * H + h) * dv + v0 + tid) * kDK;
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(lane_addr(tbase, warp, kColS + cb * 32), x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[cb * 32 + j] = x[j];
            }
        }
    } else if (tid == 0) {
        // wait (bounded) for copies this CTA still has in flight
        for (int cc = c; cc < kq_issued; ++cc) mbar_wait(&s->bar_kq[cc & 1], (cc >> 1) & 1, kWaitLimitNs);
        for (int cc = c; cc < v_issued; ++cc) mbar_wait(&s->bar_v, cc & 1, kWaitLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over [tokens][H][d] bf16, box = 64 tokens x 1 head x 64 features.
bool make_map(CUtensorMap *m, const void *base, long tokens, int H, int d)
{
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t gdim[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t gstr[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim, gstr, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gdn_tc_supported(const GdnArgs &a)
{
    const long tokens = a.cu_seqlens ? (long)a.T : (long)a.N * a.T;
    return a.dtype == 1 && a.dk == kDK && a.dv % kDVT == 0 && a.C == kC && tokens > 0 &&
           tokens < (1L << 31) && encoder() != nullptr;
}

cudaError_t gdn_launch_tc(const GdnArgs &a, cudaStream_t s, int *launches)
{
    const long tokens = a.cu_seqlens ? (long)a.T : (long)a.N * a.T;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, tokens, a.H, a.dk) || !make_map(&mk, a.k, tokens, a.H, a.dk) ||
        !make_map(&mv, a.v, tokens, a.H, a.dv))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(a.dv / kDVT, a.H, a.N);
    gdn_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, mq, mk, mv);
    *launches = 1;
    return cudaGetLastError();
}
