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

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned(const void *p, size_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

gdn_status_t chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, const float *eta, const float *S0, void *o,
                       float *S_final, int B, int H, int T, int d_k, int d_v, int C,
                       const int32_t *cu_seqlens, gdn_dtype_t dtype, void *stream)
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
    if (!any_units) return GDN_OK;
    if (!work && !S_final) return GDN_OK;  // nothing to compute, nothing to write

    GdnArgs a;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.eta = eta; a.S0 = S0;
    a.o = o; a.S_final = S_final;
    a.N = B; a.H = H; a.T = T; a.dk = d_k; a.dv = d_v; a.C = C;
    a.cu_seqlens = cu_seqlens;
    a.dtype = dtype == GDN_BF16 ? 1 : 0;
    gdn_status_t st = status_word(&a.status);
    if (st != GDN_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    cudaError_t e;
    int path;
    if (gdn_tc_supported(a)) {
        e = gdn_launch_tc(a, s, &launches);
        path = 1;
    } else {
        e = gdn_launch_simt(a, s, &launches);
        path = 0;
    }
    if (e != cudaSuccess)
        return fail(GDN_ERR_CUDA, "kernel launch (%s path): %s",
                    path ? "tcgen05" : "fp32", cudaGetErrorString(e));
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
