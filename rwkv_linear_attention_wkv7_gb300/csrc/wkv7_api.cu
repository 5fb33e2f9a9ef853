// C ABI of libwkv7: argument checking, error reporting and kernel dispatch.
// Integer status, no exit and no printing, as the extern "C" entries of the
// "Foundry/cuda_kernels/timemix.cu" page (timemix_forward_cuda) return -1 on
// failure instead of aborting.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "wkv7.h"
#include "wkv7_internal.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptr(const void *p, const char *name, bool required) {
    if (!p) return required ? fail(WKV7_EINVAL, "%s is NULL", name) : WKV7_OK;
    if (!aligned16(p)) return fail(WKV7_EINVAL, "%s is not 16-byte aligned", name);
    return WKV7_OK;
}

// The kernels are built for sm_103a only; refuse other devices up front.
int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(WKV7_EUNSUPPORTED, "no CUDA device available");
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(WKV7_EUNSUPPORTED, "cannot query device %d", dev);
    }
    if (major != 10 || minor != 3)
        return fail(WKV7_EUNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
    return WKV7_OK;
}

int check_dims(int B, int T, int H, int N, int dtype) {
    if (N != WKV7_HEAD_SIZE) return fail(WKV7_EINVAL, "N must be %d (got %d)", WKV7_HEAD_SIZE, N);
    if (B < 1 || H < 1) return fail(WKV7_EINVAL, "B and H must be >= 1 (got B=%d, H=%d)", B, H);
    if (T < 0) return fail(WKV7_EINVAL, "T must be >= 0 (got %d)", T);
    if (dtype != WKV7_F32 && dtype != WKV7_BF16) return fail(WKV7_EINVAL, "unknown dtype %d", dtype);
    if ((long long)B * H > 0x7fffffffLL) return fail(WKV7_EINVAL, "B*H too large");
    return WKV7_OK;
}

#define TRY(x)                    \
    do {                          \
        int rc_ = (x);            \
        if (rc_ != WKV7_OK) return rc_; \
    } while (0)

int launch_status(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(WKV7_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return WKV7_OK;
}

// Copy (or zero) a [B][H][N][N] state when no token is processed.
int copy_state(const float *src, float *dst, int B, int H, cudaStream_t st) {
    if (!dst) return WKV7_OK;
    const size_t bytes = (size_t)B * H * WKV7_HEAD_SIZE * WKV7_HEAD_SIZE * sizeof(float);
    cudaError_t e = src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(dst, 0, bytes, st);
    return launch_status(e, "state copy");
}

}  // namespace

// Set by a kernel whose bounded wait on its bulk copies ran out (see
// wkv7_async_status); one flag per device.
static __device__ unsigned g_async_err;
static std::mutex g_flag_mu;
static unsigned *g_flag_ptr[64] = {};

namespace wkv7 {
int set_error(int code, const char *msg) { return fail(code, "%s", msg); }

int forward_state(int B, int T, int H, int dtype, const void *w, const void *k, const void *v, const void *a,
                  const void *b, const float *s0, float *sT, int state_only, cudaStream_t st) {
    SeqArgs p{};
    p.B = B; p.T = T; p.H = H; p.L = 16; p.nck = wkv7_ckpt_count(T, 16); p.dtype = dtype;
    p.r = w; p.w = w; p.k = state_only == 1 ? k : w; p.v = state_only == 1 ? v : w; p.a = a; p.b = b;  // unread rows: any valid map
    p.s0 = s0; p.sT = sT; p.state_only = state_only;
    if (!(p.err = async_error_flag())) return WKV7_ECUDA;
    return launch_status(launch_forward_chunk(p, st), "segment pass launch");
}

int backward_state(int B, int T, int H, int dtype, const void *r, const void *w, const void *a, const void *b,
                   const float *factors, const float *dy, const float *dsT, float *ds0, cudaStream_t st) {
    SeqArgs p{};
    p.B = B; p.T = T; p.H = H; p.L = 16; p.nck = wkv7_ckpt_count(T, 16); p.dtype = dtype;
    p.r = r; p.w = w; p.k = w; p.v = w; p.a = a; p.b = b;  // k and v are not read: any valid map
    p.fac_in = factors; p.dy = dy; p.dsT = dsT; p.ds0 = ds0; p.state_only = 1;
    if (!(p.err = async_error_flag())) return WKV7_ECUDA;
    return launch_status(launch_backward_state(p, st), "state-gradient pass launch");
}

int check_call(int B, int T, int H, int N, int dtype, const void *const *req, const char *const *req_names, int nreq,
               const void *const *opt, const char *const *opt_names, int nopt) {
    TRY(check_dims(B, T, H, N, dtype));
    for (int i = 0; i < nreq; ++i) TRY(check_ptr(req[i], req_names[i], T > 0));
    for (int i = 0; i < nopt; ++i) TRY(check_ptr(opt[i], opt_names[i], false));
    return check_device();
}

unsigned *async_error_flag() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        fail(WKV7_ECUDA, "cannot identify the current device");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_flag_mu);
    if (!g_flag_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_async_err);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            fail(WKV7_ECUDA, "device error flag lookup failed: %s", cudaGetErrorString(e));
            return nullptr;
        }
        g_flag_ptr[dev] = static_cast<unsigned *>(p);
    }
    return g_flag_ptr[dev];
}
}  // namespace wkv7

extern "C" {

int wkv7_ckpt_count(int T, int L) {
    if (T < 0 || L < 1) return -1;
    return (int)(((long long)T + L - 1) / L);
}

long long wkv7_factor_floats(int T) {
    if (T < 0) return -1;
    return (((long long)T + 15) / 16) * wkv7::fac::kWords;
}

const char *wkv7_last_error(void) { return g_err; }

int wkv7_async_status(void) {
    g_err[0] = '\0';
    TRY(check_device());
    unsigned *flag = wkv7::async_error_flag();
    if (!flag) return WKV7_ECUDA;
    unsigned v = 0;
    cudaError_t e = cudaMemcpy(&v, flag, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return launch_status(e, "wkv7_async_status");
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpy(flag, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return launch_status(e, "wkv7_async_status");
        return fail(WKV7_ECUDA, "a kernel's bounded wait on its bulk copies ran out; the results of that call are invalid");
    }
    return WKV7_OK;
}

}  // extern "C"

namespace {
// The output epilogue's arguments (wkv7_forward_gn / wkv7_backward_gn); all NULL otherwise.
struct GnArgs {
    const float *gn_w = nullptr, *gn_b = nullptr, *r_k = nullptr;
    float *o = nullptr;                                          // forward
    const float *y = nullptr;                                    // backward: the forward's y
    float *dgn_w = nullptr, *dgn_b = nullptr, *dr_k = nullptr, *ws = nullptr;
    bool partials_only = false;  // backward: leave the per-(b, h) sums in ws, no reduction over batch rows
};

// prod = 1: w, a, b carry (w_pre, kk, avec) and the backward writes (dw_pre, dkk, davec)
int forward_impl(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                 const void *v, const void *a, const void *b, const float *s0, float *y, float *sT, float *ckpt,
                 float *factors, int L, void *stream, int prod, const GnArgs &gn = GnArgs()) {
    g_err[0] = '\0';
    TRY(check_dims(B, T, H, N, dtype));
    if (L < 1) return fail(WKV7_EINVAL, "L must be >= 1 (got %d)", L);
    if (factors && L != 16) return fail(WKV7_EINVAL, "factors need L == 16 (got %d)", L);
    if (prod && L % 16 != 0) return fail(WKV7_EUNSUPPORTED, "the fused producers need L a multiple of 16 (got %d)", L);
    const bool epi = gn.gn_w || gn.gn_b || gn.r_k || gn.o;
    if (epi && L % 16 != 0) return fail(WKV7_EUNSUPPORTED, "the fused epilogue needs L a multiple of 16 (got %d)", L);
    if (epi) {
        TRY(check_ptr(gn.gn_w, "gn_w", T > 0)); TRY(check_ptr(gn.gn_b, "gn_b", T > 0));
        TRY(check_ptr(gn.r_k, "r_k", T > 0)); TRY(check_ptr(gn.o, "o", T > 0));
    }
    const bool need = T > 0;
    TRY(check_ptr(r, "r", need)); TRY(check_ptr(w, prod ? "w_pre" : "w", need)); TRY(check_ptr(k, "k", need));
    TRY(check_ptr(v, "v", need)); TRY(check_ptr(a, prod ? "kk" : "a", need)); TRY(check_ptr(b, prod ? "avec" : "b", need));
    TRY(check_ptr(s0, "s0", false)); TRY(check_ptr(y, "y", need));
    TRY(check_ptr(sT, "sT", false)); TRY(check_ptr(ckpt, "ckpt", false));
    TRY(check_ptr(factors, "factors", false));
    TRY(check_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    if (T == 0) return copy_state(s0, sT, B, H, st);

    wkv7::SeqArgs p{};
    p.B = B; p.T = T; p.H = H; p.L = L; p.nck = wkv7_ckpt_count(T, L); p.dtype = dtype;
    p.r = r; p.w = w; p.k = k; p.v = v; p.a = a; p.b = b;
    p.s0 = s0; p.y = y; p.sT = sT; p.ckpt = ckpt; p.fac = factors; p.prod = prod;
    p.gn_w = gn.gn_w; p.gn_b = gn.gn_b; p.r_k = gn.r_k; p.o = gn.o;
    if (!(p.err = wkv7::async_error_flag())) return WKV7_ECUDA;
    if (wkv7::forward_chunk_supported(p)) return launch_status(wkv7::launch_forward_chunk(p, st), "wkv7_forward launch");
    return launch_status(wkv7::launch_forward_plain(p, st), "wkv7_forward launch");
}

int backward_impl(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                  const void *v, const void *a, const void *b, const float *ckpt, const float *factors, int L,
                  const float *dy, const float *dsT, float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                  float *ds0, void *stream, int prod, const GnArgs &gn = GnArgs()) {
    g_err[0] = '\0';
    TRY(check_dims(B, T, H, N, dtype));
    if (L < 1) return fail(WKV7_EINVAL, "L must be >= 1 (got %d)", L);
    if (factors && L != 16) return fail(WKV7_EINVAL, "factors need L == 16 (got %d)", L);
    const bool need = T > 0;
    if (prod && need && (L != 16 || !factors))
        return fail(WKV7_EINVAL, "the fused producers' backward needs L == 16 and the forward's factor cache");
    TRY(check_ptr(r, "r", need)); TRY(check_ptr(w, prod ? "w_pre" : "w", need)); TRY(check_ptr(k, "k", need));
    TRY(check_ptr(v, "v", need)); TRY(check_ptr(a, prod ? "kk" : "a", need)); TRY(check_ptr(b, prod ? "avec" : "b", need));
    TRY(check_ptr(ckpt, "ckpt", need)); TRY(check_ptr(factors, "factors", false));
    TRY(check_ptr(dy, "dy", need)); TRY(check_ptr(dsT, "dsT", false));
    TRY(check_ptr(dr, "dr", need)); TRY(check_ptr(dw, prod ? "dw_pre" : "dw", need)); TRY(check_ptr(dk, "dk", need));
    TRY(check_ptr(dv, "dv", need)); TRY(check_ptr(da, prod ? "dkk" : "da", need));
    TRY(check_ptr(db, prod ? "davec" : "db", need));
    TRY(check_ptr(ds0, "ds0", false));
    const bool epi = gn.gn_w != nullptr;
    if (epi) {
        if (need && (L != 16 || !factors))
            return fail(WKV7_EINVAL, "the fused epilogue's backward needs L == 16 and the forward's factor cache");
        TRY(check_ptr(gn.y, "y", need)); TRY(check_ptr(gn.gn_w, "gn_w", true)); TRY(check_ptr(gn.r_k, "r_k", true));
        TRY(check_ptr(gn.dgn_w, "dgn_w", !gn.partials_only)); TRY(check_ptr(gn.dgn_b, "dgn_b", !gn.partials_only));
        TRY(check_ptr(gn.dr_k, "dr_k", !gn.partials_only)); TRY(check_ptr(gn.ws, "workspace", true));
    }
    TRY(check_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    if (T == 0) {
        if (epi) {  // no token: the parameter gradients are zero
            const size_t bytes = (size_t)H * WKV7_HEAD_SIZE * sizeof(float);
            TRY(launch_status(cudaMemsetAsync(gn.dgn_w, 0, bytes, st), "dgn_w"));
            TRY(launch_status(cudaMemsetAsync(gn.dgn_b, 0, bytes, st), "dgn_b"));
            TRY(launch_status(cudaMemsetAsync(gn.dr_k, 0, bytes, st), "dr_k"));
        }
        return copy_state(dsT, ds0, B, H, st);
    }

    wkv7::SeqArgs p{};
    p.B = B; p.T = T; p.H = H; p.L = L; p.nck = wkv7_ckpt_count(T, L); p.dtype = dtype;
    p.r = r; p.w = w; p.k = k; p.v = v; p.a = a; p.b = b;
    p.ckpt_in = ckpt; p.fac_in = factors; p.dy = dy; p.dsT = dsT;
    p.dr = dr; p.dw = dw; p.dk = dk; p.dv = dv; p.da = da; p.db = db; p.ds0 = ds0; p.prod = prod;
    p.gn_w = gn.gn_w; p.r_k = gn.r_k; p.y_in = gn.y; p.gn_part = gn.ws;
    if (!(p.err = wkv7::async_error_flag())) return WKV7_ECUDA;
    if (epi) {
        TRY(launch_status(wkv7::launch_backward_chunk(p, st), "wkv7_backward_gn launch"));
        if (gn.partials_only) return WKV7_OK;
        return launch_status(wkv7::launch_gn_param_reduce(B, H, gn.ws, gn.dgn_w, gn.dgn_b, gn.dr_k, st),
                             "wkv7_backward_gn parameter reduction");
    }
    if (wkv7::backward_chunk_supported(p)) return launch_status(wkv7::launch_backward_chunk(p, st), "wkv7_backward launch");
    return launch_status(wkv7::launch_backward_plain(p, st), "wkv7_backward launch");
}
}  // namespace

extern "C" {

int wkv7_forward_state(int B, int T, int H, int N, wkv7_dtype dtype, const void *w, const void *k, const void *v,
                       const void *a, const void *b, const float *s0, float *sT, void *stream) {
    g_err[0] = '\0';
    TRY(check_dims(B, T, H, N, dtype));
    TRY(check_ptr(sT, "sT", true));
    TRY(check_ptr(w, "w", T > 0)); TRY(check_ptr(a, "a", T > 0)); TRY(check_ptr(b, "b", T > 0));
    TRY(check_ptr(k, "k", T > 0 && v)); TRY(check_ptr(v, "v", false)); TRY(check_ptr(s0, "s0", false));
    TRY(check_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    if (T == 0) return copy_state(s0, sT, B, H, st);
    return wkv7::forward_state(B, T, H, dtype, w, v ? k : w, v ? v : w, a, b, s0, sT, v ? 1 : 2, st);
}

int wkv7_backward_state(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *a,
                        const void *b, const float *factors, const float *dy, const float *dsT, float *ds0,
                        void *stream) {
    g_err[0] = '\0';
    TRY(check_dims(B, T, H, N, dtype));
    TRY(check_ptr(ds0, "ds0", true));
    TRY(check_ptr(r, "r", T > 0)); TRY(check_ptr(w, "w", T > 0)); TRY(check_ptr(a, "a", T > 0));
    TRY(check_ptr(b, "b", T > 0)); TRY(check_ptr(factors, "factors", T > 0)); TRY(check_ptr(dy, "dy", T > 0));
    TRY(check_ptr(dsT, "dsT", false));
    TRY(check_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    if (T == 0) return copy_state(dsT, ds0, B, H, st);
    return wkv7::backward_state(B, T, H, dtype, r, w, a, b, factors, dy, dsT, ds0, st);
}

int wkv7_forward(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                 const void *v, const void *a, const void *b, const float *s0, float *y, float *sT, float *ckpt,
                 float *factors, int L, void *stream) {
    return forward_impl(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, ckpt, factors, L, stream, 0);
}

int wkv7_backward(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                  const void *v, const void *a, const void *b, const float *ckpt, const float *factors, int L,
                  const float *dy, const float *dsT, float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                  float *ds0, void *stream) {
    return backward_impl(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, factors, L, dy, dsT, dr, dw, dk, dv, da, db,
                         ds0, stream, 0);
}

int wkv7_forward_fused(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w_pre,
                       const void *k, const void *v, const void *kk, const void *avec, const float *s0, float *y,
                       float *sT, float *ckpt, float *factors, int L, void *stream) {
    return forward_impl(B, T, H, N, dtype, r, w_pre, k, v, kk, avec, s0, y, sT, ckpt, factors, L, stream, 1);
}

int wkv7_backward_fused(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w_pre,
                        const void *k, const void *v, const void *kk, const void *avec, const float *ckpt,
                        const float *factors, int L, const float *dy, const float *dsT, float *dr, float *dw_pre,
                        float *dk, float *dv, float *dkk, float *davec, float *ds0, void *stream) {
    return backward_impl(B, T, H, N, dtype, r, w_pre, k, v, kk, avec, ckpt, factors, L, dy, dsT, dr, dw_pre, dk, dv,
                         dkk, davec, ds0, stream, 1);
}

long long wkv7_gn_workspace_floats(int B, int H) {
    if (B < 1 || H < 1) return -1;
    return (long long)B * H * 3 * WKV7_HEAD_SIZE;
}

int wkv7_forward_gn(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                    const void *v, const void *a, const void *b, const float *s0, const float *gn_w,
                    const float *gn_b, const float *r_k, float *y, float *o, float *sT, float *ckpt, float *factors,
                    int L, void *stream) {
    GnArgs gn;
    gn.gn_w = gn_w; gn.gn_b = gn_b; gn.r_k = r_k; gn.o = o;
    if (T > 0 && !(gn_w && gn_b && r_k && o)) {
        g_err[0] = '\0';
        return fail(WKV7_EINVAL, "gn_w, gn_b, r_k and o are required");
    }
    return forward_impl(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, ckpt, factors, L, stream, 0, gn);
}

int wkv7_backward_gn(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                     const void *v, const void *a, const void *b, const float *ckpt, const float *factors, int L,
                     const float *y, const float *do_, const float *dsT, const float *gn_w, const float *r_k,
                     float *dr, float *dw, float *dk, float *dv, float *da, float *db, float *ds0, float *dgn_w,
                     float *dgn_b, float *dr_k, float *workspace, void *stream) {
    GnArgs gn;
    gn.gn_w = gn_w; gn.r_k = r_k; gn.y = y; gn.dgn_w = dgn_w; gn.dgn_b = dgn_b; gn.dr_k = dr_k; gn.ws = workspace;
    if (!gn_w) {
        g_err[0] = '\0';
        return fail(WKV7_EINVAL, "gn_w is NULL");
    }
    return backward_impl(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, factors, L, do_, dsT, dr, dw, dk, dv, da, db, ds0,
                         stream, 0, gn);
}

}  // extern "C"

namespace wkv7 {
// wkv7_backward_gn without the reduction over batch rows: the per-(b, h)
// parameter-gradient sums stay in `workspace` (rows [B][H][3][N]) for a
// caller that runs launch_gn_param_reduce over more rows than this call's.
int backward_gn_partials(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                         const void *v, const void *a, const void *b, const float *ckpt, const float *factors,
                         const float *y, const float *do_, const float *dsT, const float *gn_w, const float *r_k,
                         float *dr, float *dw, float *dk, float *dv, float *da, float *db, float *ds0,
                         float *workspace, void *stream) {
    GnArgs gn;
    gn.gn_w = gn_w; gn.r_k = r_k; gn.y = y; gn.ws = workspace; gn.partials_only = true;
    if (!gn_w) {
        g_err[0] = '\0';
        return fail(WKV7_EINVAL, "gn_w is NULL");
    }
    return backward_impl(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, factors, 16, do_, dsT, dr, dw, dk, dv, da, db, ds0,
                         stream, 0, gn);
}
}  // namespace wkv7

extern "C" {

int wkv7_decode_step(int B, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                     const void *v, const void *a, const void *b, float *state, float *y, void *stream) {
    g_err[0] = '\0';
    TRY(check_dims(B, 1, H, N, dtype));
    TRY(check_ptr(r, "r", true)); TRY(check_ptr(w, "w", true)); TRY(check_ptr(k, "k", true));
    TRY(check_ptr(v, "v", true)); TRY(check_ptr(a, "a", true)); TRY(check_ptr(b, "b", true));
    TRY(check_ptr(state, "state", true)); TRY(check_ptr(y, "y", true));
    TRY(check_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    return launch_status(wkv7::launch_decode_step(B, H, dtype, r, w, k, v, a, b, state, y, st),
                         "wkv7_decode_step launch");
}

}  // extern "C"
