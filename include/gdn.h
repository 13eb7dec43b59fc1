/*
 * gdn.h — C ABI of libgdn: the chunkwise-parallel forward pass of the gated
 * delta rule on one NVIDIA GB300 (sm_103a).
 *
 * The operation (north-star recurrence; "从零开始的 GDN 推导", §"Gated Delta
 * Rule Chunk-wise Parallel 前向推导", recurrent form, written here with column
 * vectors so that the state S is d_v x d_k):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t
 *
 * evaluated chunk by chunk with the WY / UT-transform form of the same page
 * (§"UT transform", §"S 的推导", §"O 的推导", §"总结"): inside a chunk of C
 * tokens everything is dense matrix algebra; only the d_v x d_k state is
 * carried from one chunk to the next ("RNN的复兴03：现代RNN的并行计算", §四:
 * parallel inside a chunk, dependent between chunks).  The result equals the
 * sequential recurrence up to floating-point rounding.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) on
 *    the current device, row-major and contiguous.  The caller allocates and
 *    owns all of them; the library keeps no reference after the call returns.
 *  - The library allocates no device memory in these calls.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream): they validate on the host, enqueue kernels and return.
 *  - On any status other than GDN_OK nothing was enqueued, and
 *    gdn_get_last_error() returns a message for the calling thread.
 *  - There is no CPU fallback: a call either runs its CUDA kernels or fails.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, overlap   */
    GDN_ERR_UNSUPPORTED = 2, /* shape or dtype outside the compiled set      */
    GDN_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed        */
    GDN_ERR_TIMEOUT = 4,     /* gdn_get_device_status: a bounded device wait
                                ran out (GDN_DEV_WAIT_TIMEOUT is among the
                                flags; the results of that call are invalid) */
    GDN_ERR_RANGE = 5        /* gdn_get_device_status: a tensor-core operand
                                left the fp16 range (GDN_DEV_F16_RANGE is
                                among the flags; results are invalid) */
} gdn_status_t;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype_t;

/* Device-side status bits returned by gdn_get_device_status(). */
#define GDN_DEV_BAD_SEQLENS 0x1u /* a cu_seqlens span was negative or past T */
#define GDN_DEV_WAIT_TIMEOUT 0x2u /* a bounded pipeline wait gave up          */
#define GDN_DEV_F16_RANGE 0x4u    /* a tensor-core operand left the fp16 range  */
#define GDN_DEV_F16_PRECISION 0x8u /* a unit's state-chain operands all stayed
                                      below 2^-10: fp16 kept few bits of them   */

/*
 * gdn_chunk_fwd — forward pass of the gated delta rule, chunkwise.
 *
 * Arguments (N = B, the number of sequences):
 *   q          [B, T, H, d_k]  dtype   queries
 *   k          [B, T, H, d_k]  dtype   keys (the method assumes nothing about
 *                                      their norm; unit norm is the usual input)
 *   v          [B, T, H, d_v]  dtype   values
 *   log_alpha  [B, T, H]       fp32    log of the decay gate alpha_t (<= 0 is
 *                                      the usual range; not required)
 *   beta       [B, T, H]       fp32    write strength beta_t (any real value;
 *                                      (0, 2) is the extended DeltaNet range)
 *   S0         [N, H, d_v, d_k] fp32   initial state per (sequence, head), or
 *                                      NULL for zeros
 *   o          [B, T, H, d_v]  dtype   output, o_t = S_t q_t (state after
 *                                      token t); must not overlap any input
 *   S_final    [N, H, d_v, d_k] fp32   state after each sequence's last token,
 *                                      or NULL if not wanted; may be exactly
 *                                      S0 (in-place carry), must not overlap
 *                                      anything else
 *   B, H, T    batch, heads, tokens per sequence
 *   d_k, d_v   key and value head dimensions
 *   C          chunk length: 16, 32 or 64
 *   cu_seqlens device int32 [N + 1] or NULL.  When given, the sequences are
 *              packed along the token axis: q/k/v/o are [1, T, H, *],
 *              log_alpha/beta are [1, T, H], B is the number of sequences N,
 *              sequence n spans tokens [cu_seqlens[n], cu_seqlens[n+1]), and
 *              T is the packed length.  Chunks never cross a sequence; each
 *              sequence starts from its own S0[n].  Spans that are negative or
 *              run past T are skipped on the device and raise
 *              GDN_DEV_BAD_SEQLENS (see gdn_get_device_status).  On the
 *              tensor-core path, up to 256 packed sequences are started
 *              longest first, whatever their order in the pack.
 *   dtype      GDN_F32 or GDN_BF16 (q, k, v and o share it).  fp32 runs in
 *              fp32 on CUDA cores.  bf16 runs on the tensor cores with fp16
 *              operands (11-bit significand) and fp32 accumulation and
 *              state.  A bf16 input converts to fp16 exactly when its
 *              magnitude lies in [2^-14, 65504]; below 2^-14 fp16 keeps fewer
 *              bits (subnormals), above 65504 it overflows.  An operand that
 *              leaves the fp16 range raises GDN_DEV_F16_RANGE; a (sequence,
 *              head) whose state chain ran entirely below 2^-10 in magnitude
 *              (e.g. v and S0 of order 1e-6) raises GDN_DEV_F16_PRECISION:
 *              the method is linear in v and S0, so scaling both up (and the
 *              results back down) avoids it
 *   stream     cudaStream_t to enqueue on
 *
 * Alignment: q, k, v, o must be aligned to 16 bytes; log_alpha, beta, S0 and
 * S_final to 4 bytes (16 bytes lets the fastest path run).
 * Supported shapes: d_k in [1, 128], d_v >= 1, C in {16, 32, 64}.  The
 * tcgen05 tensor-core kernel serves bf16 with C = 64 and d_k, d_v multiples
 * of 8 (tiles zero-padded to 128); every other supported shape runs on the
 * fp32 CUDA-core kernel (gdn_last_launch_count reports which ran).  Both are CUDA kernels
 * of this library.
 *
 * Returns GDN_OK once the work is enqueued, or an error status (nothing
 * enqueued).  Errors detected by the kernels are reported through
 * gdn_get_device_status().
 */
gdn_status_t gdn_chunk_fwd(const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta,
                           const float *S0, void *o, float *S_final,
                           int B, int H, int T, int d_k, int d_v, int C,
                           const int32_t *cu_seqlens, gdn_dtype_t dtype,
                           void *stream);

/*
 * gdn_chunk_fwd_eta — gdn_chunk_fwd with a write strength eta_t separate
 * from the erase strength beta_t ("RNN的复兴03：现代RNN的并行计算", §一, the
 * general delta-rule recurrence):
 *
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + eta_t v_t k_t^T
 *
 * In the chunk form only U changes, U = T diag(eta) V; A and W keep beta.
 * With eta = beta this is gdn_chunk_fwd.  eta is fp32 [B, T, H] (the layout
 * of beta), non-NULL when there is work, 4-byte aligned and not overlapping
 * o or S_final.  Every other argument, and every rule, is gdn_chunk_fwd's.
 */
gdn_status_t gdn_chunk_fwd_eta(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, const float *eta,
                               const float *S0, void *o, float *S_final,
                               int B, int H, int T, int d_k, int d_v, int C,
                               const int32_t *cu_seqlens, gdn_dtype_t dtype,
                               void *stream);

/*
 * gdn_chunk_fwd_scan — gdn_chunk_fwd for few, long sequences: each sequence
 * is cut into `segments` pieces at chunk boundaries that run in parallel.
 * A segment's final state is an affine function of its initial state,
 * S_end = S_start M + B ("从零开始的 GDN 推导", §"S 的推导": every chunk step is
 * affine in S), and affine maps compose associatively ("Параллельность
 * RNN?", §"Уровень 2: рекуррентность линейна, и потому ассоциативна"): a
 * first pass computes every segment's M (d_k x d_k) and B (d_v x d_k) on the
 * tensor cores, a scan chains them into each segment's initial state, and a
 * second pass runs every segment's forward pass from it.  The result equals
 * gdn_chunk_fwd up to rounding; the work is about 2 + d_k / d_v times the
 * forward pass, spread over B * H * segments units instead of B * H.
 *
 * Arguments as gdn_chunk_fwd, packed sequences (cu_seqlens) included, plus
 *   segments   pieces per sequence; <= 0 lets the library choose from the
 *              device's SM count and the (average) sequence length (1 means
 *              the plain pass).  Without cu_seqlens it is capped at
 *              ceil(T / C) and no piece is empty.  With cu_seqlens every
 *              sequence is cut into the same number of pieces of
 *              ceil(chunks_n / segments) chunks, capped at the chunks of
 *              the whole pack; a sequence shorter than that many chunks
 *              leaves its last pieces empty.  A span that is negative or
 *              runs past T raises GDN_DEV_BAD_SEQLENS; that sequence's
 *              outputs are not written and its S_final is its S0.
 *   workspace  device scratch of at least
 *              gdn_chunk_fwd_scan_workspace_size(B, H, T, d_k, d_v, C,
 *              cu_seqlens, segments) bytes (only whether cu_seqlens is NULL
 *              matters there), 256-byte aligned, caller-owned, not
 *              overlapping any argument; NULL is allowed when that size is 0
 *              or one segment is chosen.  Calls that share a workspace must
 *              not overlap in time.
 * Supported: bf16, C = 64, d_k <= 128 and d_k, d_v multiples of 8 (the
 * tensor-core kernel); anything else returns GDN_ERR_UNSUPPORTED.  Four
 * kernels are enqueued (gdn_last_launch_count reports path 3) plus one
 * device-to-device copy per sequence for S_final.
 */
size_t gdn_chunk_fwd_scan_workspace_size(int B, int H, int T, int d_k, int d_v, int C,
                                         const int32_t *cu_seqlens, int segments);

gdn_status_t gdn_chunk_fwd_scan(const void *q, const void *k, const void *v,
                                const float *log_alpha, const float *beta,
                                const float *S0, void *o, float *S_final,
                                int B, int H, int T, int d_k, int d_v, int C,
                                const int32_t *cu_seqlens, gdn_dtype_t dtype, int segments,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_chunk_fwd_scan_noalloc — gdn_chunk_fwd_scan for callers that cannot
 * allocate device memory: the scratch is a fixed 32 MiB array that is part of
 * the library's device image (reserved when the library's module is loaded
 * on a device), so the call allocates nothing.  The pages have no
 * counterpart: this is a deployment convenience around the same scan.
 *
 * Arguments and results as gdn_chunk_fwd_scan without the workspace.  A
 * problem whose scratch (gdn_chunk_fwd_scan_workspace_size with the same
 * arguments) exceeds 32 MiB is rejected with GDN_ERR_UNSUPPORTED and a
 * message; fewer segments need less.  Nothing in the scratch has to start
 * at zero (each call writes every byte it reads).  The scratch is shared by
 * every call on a device: calls that overlap in time (other streams, other
 * threads) race and must be serialised by the caller.
 */
gdn_status_t gdn_chunk_fwd_scan_noalloc(const void *q, const void *k, const void *v,
                                        const float *log_alpha, const float *beta,
                                        const float *S0, void *o, float *S_final,
                                        int B, int H, int T, int d_k, int d_v, int C,
                                        const int32_t *cu_seqlens, gdn_dtype_t dtype,
                                        int segments, void *stream);

/*
 * gdn_decode_step — the same recurrence evaluated token by token, for decoding
 * ("从零开始的 GDN 推导", recurrent form of the gated delta rule;
 * "RNN的复兴03：现代RNN的并行计算", §一, delta-rule update), batched over
 * (sequence, head).  Per token, with r = S k:
 *
 *     S <- alpha S + beta (v - alpha r) k^T      o = S q
 *
 * which is the spec update alpha S (I - beta k k^T) + beta v k^T
 * rearranged.  T is the number of tokens each sequence advances in this call
 * (1 for one decoding step); the state stays on chip between them.  The
 * state written by gdn_chunk_fwd (S_final) is the state this call reads, so a
 * prefill with gdn_chunk_fwd followed by decode steps reproduces the
 * recurrence over the whole sequence.
 *
 * Arguments:
 *   q, k       [N, T, H, d_k]  dtype   queries, keys
 *   v          [N, T, H, d_v]  dtype   values
 *   log_alpha  [N, T, H]       fp32    log of the decay gate
 *   beta       [N, T, H]       fp32    write strength (any real value)
 *   S_in       [N, H, d_v, d_k] fp32   state before the first token, or NULL
 *                                      for zeros
 *   o          [N, T, H, d_v]  dtype   outputs; must not overlap anything
 *   S_out      [N, H, d_v, d_k] fp32   state after the last token (required);
 *                                      may be exactly S_in (in-place update),
 *                                      must not overlap anything else.  With
 *                                      T = 0 it receives S_in (or zeros).
 *   N, H, T, d_k, d_v  sizes; d_k in [1, 128], d_v >= 1
 *   dtype      GDN_F32 or GDN_BF16 (q, k, v and o share it); arithmetic is
 *              fp32 on CUDA cores either way
 *   stream     cudaStream_t to enqueue on
 *
 * Alignment: q, k, v, o 16 bytes; log_alpha, beta, S_in, S_out 4 bytes
 * (16 bytes and d_k a multiple of 4 select the vectorised kernel).
 * Returns GDN_OK once the work is enqueued (one kernel; gdn_last_launch_count
 * reports path 2), or an error status with nothing enqueued.
 */
gdn_status_t gdn_decode_step(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta,
                             const float *S_in, void *o, float *S_out,
                             int N, int H, int T, int d_k, int d_v,
                             gdn_dtype_t dtype, void *stream);

/*
 * gdn_ut_inverse — batched UT transform inverse T = (I + A)^{-1} of the
 * chunk form ("从零开始的 GDN 推导", §"UT transform") for strictly lower C x C
 * matrices A, by one of two methods, for comparing them:
 *   method 0  blocked forward substitution on CUDA cores in fp32 (the
 *             routine the tensor-core chunk kernel runs per chunk;
 *             "RNN的复兴03：现代RNN的并行计算", §2.3.1);
 *   method 1  the nilpotent doubling product on the tensor cores:
 *             (I + A)^{-1} = (I - A)(I + A^2)(I + A^4)...(I + A^32) (the
 *             finite Neumann series of the same page, §2.3.2), powers in
 *             fp16 operands, products accumulated in fp32.
 * A  [count, C, C] fp32 row-major; entries on and above the diagonal are
 *    ignored.  T [count, C, C] fp32: unit diagonal, zeros above; must not
 *    overlap A.  C in {16, 32, 64}.  One kernel; gdn_last_launch_count
 *    reports path 4 + method.  A timed-out wait of method 1 raises
 *    GDN_DEV_WAIT_TIMEOUT.
 */
gdn_status_t gdn_ut_inverse(const float *A, float *T, int count, int C, int method, void *stream);

/*
 * gdn_get_device_status — synchronise `stream`, then read and clear the
 * device-side status bits (GDN_DEV_*) raised by kernels of this library on the
 * current device since the last read.  *flags receives the bits (0 = clean).
 * Returns GDN_ERR_TIMEOUT when GDN_DEV_WAIT_TIMEOUT is among them (*flags is
 * still written): a kernel gave up on a bounded wait, finished without
 * completing its work, drained what it had in flight and freed its tensor
 * memory, so the device stays usable but that work's outputs are invalid.
 * Else GDN_ERR_RANGE when GDN_DEV_F16_RANGE is among them: an operand
 * overflowed fp16, so the outputs it fed are wrong.  The other bits (a bad
 * packed span: that sequence was skipped; fp16 precision: results are valid
 * but carry fewer bits) come back with GDN_OK.
 * Returns GDN_ERR_CUDA if synchronising or reading fails.
 */
gdn_status_t gdn_get_device_status(void *stream, unsigned int *flags);

/* Message for the last non-OK status returned on the calling thread. */
const char *gdn_get_last_error(void);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int gdn_version(void);

/*
 * gdn_last_launch_count — number of kernels the last successful gdn_chunk_fwd
 * gdn_chunk_fwd_scan or gdn_decode_step on the calling thread enqueued, and
 * in *path which kernel family ran (0 = fp32 CUDA-core chunk kernel,
 * 1 = tcgen05 tensor-core chunk kernel, 2 = recurrent decode kernel,
 * 3 = chunk-level scan over segments, 4 / 5 = UT inverse by forward
 * substitution / on the tensor cores).  For
 * accounting in benchmarks; no device work.
 */
int gdn_last_launch_count(int *path);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
