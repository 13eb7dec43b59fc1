// C-ABI front end of libgdn: argument validation, kernel selection, and the
// device status word.  See include/gdn.h for the contract of each entry point.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char t_msg[512] = "";
thread_local int t_launches = 0;
thread_local int t_path = -1;

// Device status word: kernels OR GDN_DEV_* bits into it; the host reads and
// clears it in gdn_get_device_status().
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
unsigned int *g_status_ptr[kMaxDevices];  // per-device address of g_status_word

// Fixed scratch of gdn_chunk_fwd_scan_noalloc: part of the library's device
// image, so the call itself allocates nothing.  Every byte the scan reads is
// written earlier in the same call (segment boundaries, start states, the
// propagators), so nothing has to start at zero; two calls in flight at the
// same time on one device share it and race.
constexpr size_t kNoAllocScratchBytes = 32u << 20;
__device__ __align__(256) unsigned char g_scan_scratch[kNoAllocScratchBytes];
void *g_scratch_ptr[kMaxDevices];  // per-device address of g_scan_scratch

gdn_status_t fail(gdn_status_t st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
    va_end(ap);
    return st;
}

gdn_status_t status_word(unsigned int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device index %d", dev);
    unsigned int *p = __atomic_load_n(&g_status_ptr[dev], __ATOMIC_ACQUIRE);
    if (!p) {
        e = cudaGetSymbolAddress((void **)&p, g_status_word);
        if (e != cudaSuccess)
            return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        __atomic_store_n(&g_status_ptr[dev], p, __ATOMIC_RELEASE);
    }
    *out = p;
    return GDN_OK;
}

gdn_status_t scan_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device index %d", dev);
    void *p = __atomic_load_n(&g_scratch_ptr[dev], __ATOMIC_ACQUIRE);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_scan_scratch);
        if (e != cudaSuccess)
            return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        __atomic_store_n(&g_scratch_ptr[dev], p, __ATOMIC_RELEASE);
    }
    *out = p;
    return GDN_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned(const void *p, size_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

// Workspace of the chunk-level scan: segment boundaries, the state each
// segment starts from, the segments' zero-start states (later their final
// states) and their d_k x d_k transitions.
struct ScanLayout {
    size_t cu, sin, bseg, mseg, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

ScanLayout scan_layout(int B, int H, int d_k, int d_v, int P)
{
    const size_t nseg = (size_t)B * P;
    ScanLayout l;
    l.cu = 0;
    l.sin = align256((nseg + 1) * sizeof(int32_t));
    l.bseg = l.sin + align256(nseg * H * d_v * d_k * sizeof(float));
    l.mseg = l.bseg + align256(nseg * H * d_v * d_k * sizeof(float));
    l.total = l.mseg + align256(nseg * H * d_k * d_k * sizeof(float));
    return l;
}

// Segments per sequence: minimise the modelled time of the propagator pass
// (d_v tiles + one identity tile per unit) and the forward pass (d_v tiles)
// over waves of clusters, plus the sequential scan (about half a chunk step
// per segment).
int choose_segments(int B, int H, int d_v, int nchunks)
{
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long slots = sms / 2 > 0 ? sms / 2 : 1;  // one 2-CTA cluster per unit and wave
    const long vt = (d_v + 127) / 128;
    int best = 1;
    double best_t = 1e300;
    for (int P = 1; P <= nchunks && P <= 4096; ++P) {
        const long per = (nchunks + P - 1) / P;
        const long w1 = ((long)B * H * P * (vt + 1) + slots - 1) / slots;
        const long w3 = ((long)B * H * P * vt + slots - 1) / slots;
        const double t = P == 1 ? (double)((B * H * vt + slots - 1) / slots) * nchunks
                                : (double)(w1 + w3) * per + 0.5 * P;
        if (t < best_t) {
            best_t = t;
            best = P;
        }
    }
    return best;
}

// Host checks of a forward-pass call; on success *a describes it (with the
// device status word) and *nothing is set when there is nothing to compute.
// Segments per sequence for a request (<= 0: chosen here), with no empty
// segment: ceil(nchunks / ceil(nchunks / P)).
int segment_count(int B, int H, int d_v, int nchunks, int segments)
{
    int P = segments > 0 ? (segments < nchunks ? segments : nchunks)
                         : choose_segments(B, H, d_v, nchunks);
    if (P < 1) P = 1;
    const int per = (nchunks + P - 1) / P;
    return (nchunks + per - 1) / per;
}

// Segments per sequence for a call: packed sequences (lengths on the device)
// are cut into the same number of segments each, chosen from the average
// length T / B when not given, and never more than the chunks of the whole
// pack; a short sequence's trailing segments are then empty.
int segment_count_for(int B, int H, int T, int d_v, int C, bool packed, int segments)
{
    if (!packed) return segment_count(B, H, d_v, (T + C - 1) / C, segments);
    const long total_chunks = ((long)T + C - 1) / C;
    const int avg = (int)((total_chunks + B - 1) / B);
    int P = segments > 0 ? segments : choose_segments(B, H, d_v, avg > 0 ? avg : 1);
    if (P > total_chunks) P = (int)total_chunks;
    return P < 1 ? 1 : P;
}

gdn_status_t check_chunk(const void *q, const void *k, const void *v, const float *log_alpha,
                         const float *beta, const float *eta, const float *S0, void *o,
                         float *S_final, int B, int H, int T, int d_k, int d_v, int C,
                         const int32_t *cu_seqlens, gdn_dtype_t dtype, GdnArgs *a, bool *nothing)
{
    t_msg[0] = '\0';
    if (B < 0 || H < 0 || T < 0)
        return fail(GDN_ERR_INVALID_ARG, "negative size: B=%d H=%d T=%d", B, H, T);
    if (d_k < 1 || d_v < 1)
        return fail(GDN_ERR_INVALID_ARG, "head dims must be >= 1: d_k=%d d_v=%d", d_k, d_v);
    if (dtype != GDN_F32 && dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "dtype %d (expected GDN_F32 or GDN_BF16)", (int)dtype);
    if (C != 16 && C != 32 && C != 64)
        return fail(GDN_ERR_UNSUPPORTED, "chunk length C=%d (supported: 16, 32, 64)", C);
    if (d_k > 128)
        return fail(GDN_ERR_UNSUPPORTED, "d_k=%d (supported: 1..128)", d_k);
    if (cu_seqlens && B < 1)
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens given with B=%d sequences", B);

    const size_t esz = dtype == GDN_BF16 ? 2 : 4;
    const size_t tokens = cu_seqlens ? (size_t)T : (size_t)B * T;  // token rows
    const size_t nqk = tokens * H * d_k * esz, nv = tokens * H * d_v * esz;
    const size_t ng = tokens * H * sizeof(float);
    const size_t ns = (size_t)B * H * d_v * d_k * sizeof(float);
    const bool work = tokens > 0 && H > 0;
    const bool any_units = (size_t)B * H > 0;

    if (work && (!q || !k || !v || !log_alpha || !beta || !o))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, log_alpha, beta and o must be non-NULL");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (!aligned(log_alpha, 4) || !aligned(beta, 4) || !aligned(eta, 4) || !aligned(S0, 4) ||
        !aligned(S_final, 4))
        return fail(GDN_ERR_INVALID_ARG,
                    "log_alpha, beta, eta, S0 and S_final must be 4-byte aligned");
    if (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv) ||
        overlaps(o, nv, log_alpha, ng) || overlaps(o, nv, beta, ng) || overlaps(o, nv, eta, ng) ||
        overlaps(o, nv, S0, ns) || overlaps(o, nv, S_final, ns))
        return fail(GDN_ERR_INVALID_ARG, "o overlaps another argument");
    if (S_final && S_final != S0 &&
        (overlaps(S_final, ns, q, nqk) || overlaps(S_final, ns, k, nqk) ||
         overlaps(S_final, ns, v, nv) || overlaps(S_final, ns, log_alpha, ng) ||
         overlaps(S_final, ns, beta, ng) || overlaps(S_final, ns, eta, ng) ||
         overlaps(S_final, ns, S0, ns)))
        return fail(GDN_ERR_INVALID_ARG, "S_final overlaps an input (only S_final == S0 is allowed)");

    t_launches = 0;
    t_path = -1;
    *nothing = !any_units || (!work && !S_final);  // nothing to compute, nothing to write
    if (*nothing) return GDN_OK;
    a->q = q; a->k = k; a->v = v; a->log_alpha = log_alpha; a->beta = beta; a->eta = eta;
    a->S0 = S0; a->o = o; a->S_final = S_final;
    a->N = B; a->H = H; a->T = T; a->dk = d_k; a->dv = d_v; a->C = C;
    a->cu_seqlens = cu_seqlens;
    a->dtype = dtype == GDN_BF16 ? 1 : 0;
    a->mode = 0;
    a->prop_M = nullptr;
    return status_word(&a->status);
}

gdn_status_t launch_chunk(const GdnArgs &a, cudaStream_t s, int *launches, int *path)
{
    cudaError_t e;
    if (gdn_tc_supported(a)) {
        e = gdn_launch_tc(a, s, launches);
        *path = 1;
    } else {
        e = gdn_launch_simt(a, s, launches);
        *path = 0;
    }
    if (e != cudaSuccess)
        return fail(GDN_ERR_CUDA, "kernel launch (%s path): %s",
                    *path ? "tcgen05" : "fp32", cudaGetErrorString(e));
    return GDN_OK;
}

gdn_status_t chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, const float *eta, const float *S0, void *o,
                       float *S_final, int B, int H, int T, int d_k, int d_v, int C,
                       const int32_t *cu_seqlens, gdn_dtype_t dtype, void *stream)
{
    GdnArgs a;
    bool nothing = false;
    gdn_status_t st = check_chunk(q, k, v, log_alpha, beta, eta, S0, o, S_final, B, H, T, d_k, d_v,
                                  C, cu_seqlens, dtype, &a, &nothing);
    if (st != GDN_OK || nothing) return st;
    int launches = 0, path = -1;
    st = launch_chunk(a, static_cast<cudaStream_t>(stream), &launches, &path);
    if (st != GDN_OK) return st;
    t_launches = launches;
    t_path = path;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_get_last_error(void) { return t_msg; }

int gdn_version(void) { return 100; }

int gdn_last_launch_count(int *path)
{
    if (path) *path = t_path;
    return t_launches;
}

gdn_status_t gdn_get_device_status(void *stream, unsigned int *flags)
{
    if (!flags) return fail(GDN_ERR_INVALID_ARG, "flags is NULL");
    unsigned int *p = nullptr;
    gdn_status_t st = status_word(&p);
    if (st != GDN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    unsigned int v = 0;
    e = cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(v), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "reading device status: %s", cudaGetErrorString(e));
    *flags = v;
    if (v & GDN_DEV_WAIT_TIMEOUT)
        return fail(GDN_ERR_TIMEOUT, "a bounded device wait ran out (flags %#x): outputs invalid", v);
    if (v & GDN_DEV_F16_RANGE)
        return fail(GDN_ERR_RANGE, "a tensor-core operand left the fp16 range (flags %#x): outputs invalid", v);
    return GDN_OK;
}

gdn_status_t gdn_chunk_fwd(const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta,
                           const float *S0, void *o, float *S_final,
                           int B, int H, int T, int d_k, int d_v, int C,
                           const int32_t *cu_seqlens, gdn_dtype_t dtype,
                           void *stream)
{
    return chunk_fwd(q, k, v, log_alpha, beta, nullptr, S0, o, S_final, B, H, T, d_k, d_v, C,
                     cu_seqlens, dtype, stream);
}

gdn_status_t gdn_chunk_fwd_eta(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, const float *eta,
                               const float *S0, void *o, float *S_final,
                               int B, int H, int T, int d_k, int d_v, int C,
                               const int32_t *cu_seqlens, gdn_dtype_t dtype,
                               void *stream)
{
    if (!eta && B > 0 && H > 0 && T > 0) {
        t_msg[0] = '\0';
        return fail(GDN_ERR_INVALID_ARG, "eta must be non-NULL (use gdn_chunk_fwd for eta = beta)");
    }
    return chunk_fwd(q, k, v, log_alpha, beta, eta, S0, o, S_final, B, H, T, d_k, d_v, C,
                     cu_seqlens, dtype, stream);
}

size_t gdn_chunk_fwd_scan_workspace_size(int B, int H, int T, int d_k, int d_v, int C,
                                         const int32_t *cu_seqlens, int segments)
{
    if (B <= 0 || H <= 0 || T <= 0 || d_k <= 0 || d_v <= 0 || (C != 16 && C != 32 && C != 64))
        return 0;
    const int P = segment_count_for(B, H, T, d_v, C, cu_seqlens != nullptr, segments);
    return P <= 1 ? 0 : scan_layout(B, H, d_k, d_v, P).total;
}

gdn_status_t gdn_chunk_fwd_scan(const void *q, const void *k, const void *v,
                                const float *log_alpha, const float *beta,
                                const float *S0, void *o, float *S_final,
                                int B, int H, int T, int d_k, int d_v, int C,
                                const int32_t *cu_seqlens, gdn_dtype_t dtype, int segments,
                                void *workspace, size_t workspace_bytes, void *stream)
{
    GdnArgs a;
    bool nothing = false;
    gdn_status_t st = check_chunk(q, k, v, log_alpha, beta, nullptr, S0, o, S_final, B, H, T, d_k,
                                  d_v, C, cu_seqlens, dtype, &a, &nothing);
    if (st != GDN_OK || nothing) return st;
    if (!gdn_tc_supported(a))
        return fail(GDN_ERR_UNSUPPORTED,
                    "the chunk-level scan runs on the tensor-core kernel: bf16, C = 64 and d_k, d_v "
                    "multiples of 8 (got dtype %d, d_k=%d, d_v=%d, C=%d)", (int)dtype, d_k, d_v, C);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int P = segment_count_for(B, H, T, d_v, C, cu_seqlens != nullptr, segments);
    int launches = 0, path = -1;
    if (P <= 1) {  // one segment per sequence: the plain forward pass
        st = launch_chunk(a, s, &launches, &path);
        if (st != GDN_OK) return st;
        t_launches = launches;
        t_path = path;
        return GDN_OK;
    }
    const ScanLayout l = scan_layout(B, H, d_k, d_v, P);
    if (!workspace || workspace_bytes < l.total)
        return fail(GDN_ERR_INVALID_ARG, "workspace of %zu bytes needed (%zu given)", l.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (!aligned(workspace, 256))
        return fail(GDN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t tokens = cu_seqlens ? (size_t)T : (size_t)B * T;
    const size_t nqk = tokens * H * d_k * 2, nv = tokens * H * d_v * 2;
    const size_t ng = tokens * H * sizeof(float), ns = (size_t)B * H * d_v * d_k * sizeof(float);
    if (overlaps(workspace, l.total, q, nqk) || overlaps(workspace, l.total, k, nqk) ||
        overlaps(workspace, l.total, v, nv) || overlaps(workspace, l.total, o, nv) ||
        overlaps(workspace, l.total, log_alpha, ng) || overlaps(workspace, l.total, beta, ng) ||
        overlaps(workspace, l.total, S0, ns) || overlaps(workspace, l.total, S_final, ns) ||
        overlaps(workspace, l.total, cu_seqlens, cu_seqlens ? (size_t)(B + 1) * sizeof(int32_t) : 0))
        return fail(GDN_ERR_INVALID_ARG, "workspace overlaps an argument");

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *cu = reinterpret_cast<int32_t *>(ws + l.cu);
    float *Sin = reinterpret_cast<float *>(ws + l.sin);
    float *Bseg = reinterpret_cast<float *>(ws + l.bseg);
    float *Mseg = reinterpret_cast<float *>(ws + l.mseg);
    // (1) segment boundaries, as packed sequences over the token rows
    cudaError_t e = gdn_launch_segments(cu, cu_seqlens, B, P, T, C, a.status, s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "segment boundaries: %s", cudaGetErrorString(e));
    // (2) propagators: per segment, the state reached from zero and the transition
    GdnArgs pa = a;
    pa.N = B * P;
    pa.T = (int)tokens;
    pa.cu_seqlens = cu;
    pa.S0 = nullptr;
    pa.S_final = Bseg;
    pa.mode = 1;
    pa.prop_M = Mseg;
    int n = 0;
    e = gdn_launch_tc(pa, s, &n);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "propagator pass: %s", cudaGetErrorString(e));
    // (3) the state each segment starts from
    e = gdn_launch_scan(S0, Bseg, Mseg, Sin, B, P, H, d_v, d_k, a.status, s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "segment scan: %s", cudaGetErrorString(e));
    // (4) the forward pass of every segment from its own start state
    GdnArgs fa = pa;
    fa.S0 = Sin;
    fa.S_final = Bseg;  // the segments' final states (the zero-start states are consumed)
    fa.mode = 0;
    fa.prop_M = nullptr;
    e = gdn_launch_tc(fa, s, &n);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "segment forward pass: %s", cudaGetErrorString(e));
    // (5) each sequence's final state is its last segment's
    if (S_final) {
        const size_t per_seq = (size_t)H * d_v * d_k * sizeof(float);
        for (int b = 0; b < B; ++b) {
            e = cudaMemcpyAsync(reinterpret_cast<uint8_t *>(S_final) + b * per_seq,
                                reinterpret_cast<uint8_t *>(Bseg) + ((size_t)b * P + P - 1) * per_seq,
                                per_seq, cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess)
                return fail(GDN_ERR_CUDA, "final state copy: %s", cudaGetErrorString(e));
        }
    }
    t_launches = 4;
    t_path = 3;
    return GDN_OK;
}

gdn_status_t gdn_chunk_fwd_scan_noalloc(const void *q, const void *k, const void *v,
                                        const float *log_alpha, const float *beta,
                                        const float *S0, void *o, float *S_final,
                                        int B, int H, int T, int d_k, int d_v, int C,
                                        const int32_t *cu_seqlens, gdn_dtype_t dtype, int segments,
                                        void *stream)
{
    t_msg[0] = '\0';
    const size_t need = gdn_chunk_fwd_scan_workspace_size(B, H, T, d_k, d_v, C, cu_seqlens, segments);
    if (need > kNoAllocScratchBytes)
        return fail(GDN_ERR_UNSUPPORTED,
                    "this problem needs %zu bytes of scan scratch; the fixed scratch holds %zu "
                    "(use gdn_chunk_fwd_scan with a workspace, or fewer segments)",
                    need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        gdn_status_t st = scan_scratch(&scratch);
        if (st != GDN_OK) return st;
    }
    return gdn_chunk_fwd_scan(q, k, v, log_alpha, beta, S0, o, S_final, B, H, T, d_k, d_v, C,
                              cu_seqlens, dtype, segments, scratch,
                              need > 0 ? kNoAllocScratchBytes : 0, stream);
}

gdn_status_t gdn_ut_inverse(const float *A, float *T, int count, int C, int method, void *stream)
{
    t_msg[0] = '\0';
    if (count < 0) return fail(GDN_ERR_INVALID_ARG, "negative count %d", count);
    if (C != 16 && C != 32 && C != 64)
        return fail(GDN_ERR_UNSUPPORTED, "C=%d (supported: 16, 32, 64)", C);
    if (method != 0 && method != 1)
        return fail(GDN_ERR_UNSUPPORTED, "method %d (0: forward substitution, 1: tensor cores)",
                    method);
    const size_t bytes = (size_t)count * C * C * sizeof(float);
    if (count > 0 && (!A || !T)) return fail(GDN_ERR_INVALID_ARG, "A and T must be non-NULL");
    if (!aligned(A, 4) || !aligned(T, 4))
        return fail(GDN_ERR_INVALID_ARG, "A and T must be 4-byte aligned");
    if (overlaps(A, bytes, T, bytes)) return fail(GDN_ERR_INVALID_ARG, "T overlaps A");
    t_launches = 0;
    t_path = -1;
    if (count == 0) return GDN_OK;
    unsigned int *status = nullptr;
    gdn_status_t st = status_word(&status);
    if (st != GDN_OK) return st;
    cudaError_t e = gdn_launch_ut_inverse(A, T, count, C, method, status,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "UT inverse launch: %s", cudaGetErrorString(e));
    t_launches = 1;
    t_path = 4 + method;
    return GDN_OK;
}

gdn_status_t gdn_decode_step(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta,
                             const float *S_in, void *o, float *S_out,
                             int N, int H, int T, int d_k, int d_v,
                             gdn_dtype_t dtype, void *stream)
{
    t_msg[0] = '\0';
    if (N < 0 || H < 0 || T < 0)
        return fail(GDN_ERR_INVALID_ARG, "negative size: N=%d H=%d T=%d", N, H, T);
    if (d_k < 1 || d_v < 1)
        return fail(GDN_ERR_INVALID_ARG, "head dims must be >= 1: d_k=%d d_v=%d", d_k, d_v);
    if (dtype != GDN_F32 && dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "dtype %d (expected GDN_F32 or GDN_BF16)", (int)dtype);
    if (d_k > 128)
        return fail(GDN_ERR_UNSUPPORTED, "d_k=%d (supported: 1..128)", d_k);

    const size_t esz = dtype == GDN_BF16 ? 2 : 4;
    const size_t tokens = (size_t)N * T;
    const size_t nqk = tokens * H * d_k * esz, nv = tokens * H * d_v * esz;
    const size_t ng = tokens * H * sizeof(float);
    const size_t ns = (size_t)N * H * d_v * d_k * sizeof(float);
    const bool any_units = (size_t)N * H > 0;
    const bool work = any_units && T > 0;

    if (any_units && !S_out) return fail(GDN_ERR_INVALID_ARG, "S_out must be non-NULL");
    if (work && (!q || !k || !v || !log_alpha || !beta || !o))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, log_alpha, beta and o must be non-NULL");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (!aligned(log_alpha, 4) || !aligned(beta, 4) || !aligned(S_in, 4) || !aligned(S_out, 4))
        return fail(GDN_ERR_INVALID_ARG, "log_alpha, beta, S_in and S_out must be 4-byte aligned");
    if (work && (overlaps(o, nv, q, nqk) || overlaps(o, nv, k, nqk) || overlaps(o, nv, v, nv) ||
                 overlaps(o, nv, log_alpha, ng) || overlaps(o, nv, beta, ng) ||
                 overlaps(o, nv, S_in, ns) || overlaps(o, nv, S_out, ns)))
        return fail(GDN_ERR_INVALID_ARG, "o overlaps another argument");
    if (S_out != S_in &&
        (overlaps(S_out, ns, q, nqk) || overlaps(S_out, ns, k, nqk) || overlaps(S_out, ns, v, nv) ||
         overlaps(S_out, ns, log_alpha, ng) || overlaps(S_out, ns, beta, ng) ||
         overlaps(S_out, ns, S_in, ns)))
        return fail(GDN_ERR_INVALID_ARG, "S_out overlaps an input (only S_out == S_in is allowed)");

    t_launches = 0;
    t_path = -1;
    if (!any_units) return GDN_OK;

    GdnDecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
    a.S_in = S_in; a.o = o; a.S_out = S_out;
    a.N = N; a.H = H; a.T = T; a.dk = d_k; a.dv = d_v;
    a.dtype = dtype == GDN_BF16 ? 1 : 0;
    int launches = 0;
    cudaError_t e = gdn_launch_decode(a, static_cast<cudaStream_t>(stream), &launches);
    if (e != cudaSuccess)
        return fail(GDN_ERR_CUDA, "kernel launch (decode): %s", cudaGetErrorString(e));
    t_launches = launches;
    t_path = 2;
    return GDN_OK;
}

}  // extern "C"
