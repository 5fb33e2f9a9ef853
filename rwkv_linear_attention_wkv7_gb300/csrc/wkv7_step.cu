// One training step of the recurrence in one call, as concurrent blocks of
// batch rows: wkv7_forward_backward (the forward with checkpoints at stride
// 16 and the factor cache, then the backward), and the same for the fused
// producers (wkv7_forward_backward_fused) and the output epilogue
// (wkv7_forward_backward_gn).
//
// Every (b, h) is independent in both directions, so the batch splits into
// nsplit contiguous blocks of rows, each running its forward and then its
// backward on a stream of its own.  A block's backward starts as soon as its
// own forward is done, while the other blocks' forward CTAs are still
// finishing.  With one CTA per head the forward leaves a tail of unevenly
// loaded SMs and the backward a partly empty second wave; the blocks fill
// each other's.
//
// Block 0 runs on the caller's stream, the others on streams of the library,
// forked from the caller's stream by an event and joined back into it, so the
// call stays stream-ordered for the caller.  Using the caller's stream for
// one block keeps the library's streams to nsplit - 1 (one for the default
// split): every extra stream can share a hardware work queue with the
// caller's other streams, such as copy streams, and serialise work they meant
// to overlap.  run_side_by_side, the fork / join itself, also runs the time
// split's two independent segment passes (wkv7_timesplit.cu).
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "wkv7.h"
#include "wkv7_internal.cuh"

namespace wkv7 {
// wkv7_backward_gn without the reduction over batch rows: the per-(b, h)
// parameter-gradient sums stay in `workspace` (wkv7_api.cu).
int backward_gn_partials(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                         const void *v, const void *a, const void *b, const float *ckpt, const float *factors,
                         const float *y, const float *do_, const float *dsT, const float *gn_w, const float *r_k,
                         float *dr, float *dw, float *dk, float *dv, float *da, float *db, float *ds0,
                         float *workspace, void *stream);
}  // namespace wkv7

namespace {

constexpr int kMaxSplit = 4;
// The default number of blocks, as measured: four once the batch has at
// least 512 heads, two below that.  bf16 T=4096 H=32, four blocks against
// two: 16 rows 3.545 and 3.565 ms, 8 rows 2.045 and 2.044, 4 rows 1.565 and
// 1.559; fp32 T=4096 H=40: 16 rows 5.874 and 5.897, 64 rows 21.383 and
// 21.395.
int default_split(int B, int H) { return (long long)B * H >= 512 ? 4 : 2; }
// Blocks a call runs (arguments already checked): one when there is no token.
int blocks_of(int B, int T, int H, int nsplit) {
    const int n = nsplit == 0 ? default_split(B, H) : nsplit;
    return T == 0 ? 1 : (n < B ? n : B);
}
constexpr int kMaxDevices = 64;

// Streams and events of one device, created when a call first needs them and
// kept for the process (slot 0 is never used: block 0 runs on the caller's
// stream).  Calls reuse the events, so each call enqueues its work while
// holding g_mu (only the enqueueing, not the execution, is serialised).
struct Pool {
    int streams = 1;  // slots 1 .. streams - 1 exist
    cudaStream_t s[kMaxSplit] = {};
    cudaEvent_t fork = nullptr, join[kMaxSplit] = {};
};
std::mutex g_mu;
Pool g_pool[kMaxDevices];

int cuda_fail(cudaError_t e, const char *what) {
    cudaGetLastError();
    char msg[200];
    snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return wkv7::set_error(WKV7_ECUDA, msg);
}

// The current device's pool with streams for blocks 1 .. n - 1 (g_mu held by
// the caller).
int pool_of_device(int n, Pool **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return wkv7::set_error(WKV7_EUNSUPPORTED, "device index beyond the stream pool");
    Pool &p = g_pool[dev];
    if (!p.fork && (e = cudaEventCreateWithFlags(&p.fork, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e, "event creation");
    for (; p.streams < n; ++p.streams) {
        const int i = p.streams;
        if ((e = cudaStreamCreateWithFlags(&p.s[i], cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "stream creation");
        if ((e = cudaEventCreateWithFlags(&p.join[i], cudaEventDisableTiming)) != cudaSuccess) {
            cudaStreamDestroy(p.s[i]);
            return cuda_fail(e, "event creation");
        }
    }
    *out = &p;
    return WKV7_OK;
}

}  // namespace

namespace wkv7 {
// Runs work(i, stream, ctx) for i = 0 .. n - 1 side by side: piece 0 on the
// caller's stream, the others on the library's streams, forked from the
// caller's stream by an event and joined back into it, also after an error.
// g_mu is held while the work is enqueued.
int run_side_by_side(int n, cudaStream_t caller, int (*work)(int, cudaStream_t, void *), void *ctx) {
    if (n < 1 || n > kMaxSplit) return set_error(WKV7_EINVAL, "run_side_by_side: 1 .. 4 pieces");
    std::lock_guard<std::mutex> lock(g_mu);
    Pool *pool = nullptr;
    int rc = pool_of_device(n, &pool);
    if (rc != WKV7_OK) return rc;
    cudaError_t e = cudaEventRecord(pool->fork, caller);
    if (e != cudaSuccess) return cuda_fail(e, "fork event");
    int joined = 1;  // library streams given work (1 .. joined - 1)
    for (int i = 0; i < n && rc == WKV7_OK; ++i) {
        cudaStream_t s = i ? pool->s[i] : caller;
        if (i) {
            if ((e = cudaStreamWaitEvent(s, pool->fork, 0)) != cudaSuccess) {
                rc = cuda_fail(e, "fork wait");
                break;
            }
            joined = i + 1;
        }
        rc = work(i, s, ctx);
    }
    for (int i = 1; i < joined; ++i) {
        const cudaError_t j1 = cudaEventRecord(pool->join[i], pool->s[i]);
        const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(caller, pool->join[i], 0) : j1;
        if (j2 != cudaSuccess && rc == WKV7_OK) rc = cuda_fail(j2, "join");
    }
    return rc;
}
}  // namespace wkv7

namespace {

// Runs block(b0, nb, stream) for n blocks of batch rows (rows b0 .. b0 + nb - 1)
// side by side (run_side_by_side).
template <typename Block>
int run_blocks(int B, int n, cudaStream_t caller, Block &&block) {
    struct Ctx {
        int B, n;
        Block *block;
    } ctx{B, n, &block};
    return wkv7::run_side_by_side(n, caller, [](int i, cudaStream_t s, void *c) -> int {
        const Ctx &x = *static_cast<const Ctx *>(c);
        const int b0 = (int)((long long)i * x.B / x.n), b1 = (int)((long long)(i + 1) * x.B / x.n);
        return (*x.block)(b0, b1 - b0, s);
    }, &ctx);
}

// Element offsets of batch row b0 in the library's layouts.
struct Rows {
    size_t esize, seq, state, ck, fac;
    Rows(int T, int H, wkv7_dtype dtype)
        : esize(dtype == WKV7_BF16 ? 2 : 4),
          seq((size_t)T * H * WKV7_HEAD_SIZE),                        // [B][T][H][N]
          state((size_t)H * WKV7_HEAD_SIZE * WKV7_HEAD_SIZE),         // [B][H][N][N]
          ck(state * (size_t)wkv7_ckpt_count(T, 16)),                 // [B][H][ceil(T/16)][N][N]
          fac((size_t)H * (size_t)wkv7_factor_floats(T)) {}           // [B][H][factor floats]
    const void *in(const void *p, int b0) const {                     // an input row, fp32 or bf16
        return p ? static_cast<const void *>(static_cast<const char *>(p) + (size_t)b0 * seq * esize) : p;
    }
    template <typename P>
    P *at(P *p, int b0, size_t row) const { return p ? p + (size_t)b0 * row : p; }
};

int check_nsplit(int nsplit) {
    if (nsplit >= 0 && nsplit <= kMaxSplit) return WKV7_OK;
    char msg[80];
    snprintf(msg, sizeof msg, "nsplit must be 0 (the default) .. %d (got %d)", kMaxSplit, nsplit);
    return wkv7::set_error(WKV7_EINVAL, msg);
}

using ForwardFn = int (*)(int, int, int, int, wkv7_dtype, const void *, const void *, const void *, const void *,
                         const void *, const void *, const float *, float *, float *, float *, float *, int, void *);
using BackwardFn = int (*)(int, int, int, int, wkv7_dtype, const void *, const void *, const void *, const void *,
                          const void *, const void *, const float *, const float *, int, const float *,
                          const float *, float *, float *, float *, float *, float *, float *, float *, void *);

// The step through a forward / backward pair of entry points with one
// signature: the plain ones, or those with the producers fused in (whose w,
// a, b slots carry w_pre, kk, avec and whose dw, da, db slots receive their
// gradients).
int step(ForwardFn fwd, BackwardFn bwd, bool fused, int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w,
         const void *k, const void *v, const void *a, const void *b, const float *s0, const float *dy,
         const float *dsT, float *y, float *sT, float *ckpt, float *factors, float *dr, float *dw, float *dk,
         float *dv, float *da, float *db, float *ds0, int nsplit, void *stream) {
    if (check_nsplit(nsplit) != WKV7_OK) return WKV7_EINVAL;
    {   // every argument is checked before the first launch
        const void *req[15] = {r, w, k, v, a, b, dy, y, ckpt, dr, dw, dk, dv, da, db};
        const char *rn_plain[15] = {"r", "w", "k", "v", "a", "b", "dy", "y", "ckpt", "dr", "dw", "dk", "dv", "da", "db"};
        const char *rn_fused[15] = {"r", "w_pre", "k", "v", "kk", "avec", "dy", "y", "ckpt",
                                    "dr", "dw_pre", "dk", "dv", "dkk", "davec"};
        const char *const *rn = fused ? rn_fused : rn_plain;
        const void *opt[5] = {s0, dsT, sT, factors, ds0};
        const char *on[5] = {"s0", "dsT", "sT", "factors", "ds0"};
        const int rc = wkv7::check_call(B, T, H, N, dtype, req, rn, 15, opt, on, 5);
        if (rc != WKV7_OK) return rc;
    }
    const int n = blocks_of(B, T, H, nsplit);
    if (n == 1) {  // one block: the two calls in order on the caller's stream
        int rc = fwd(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, ckpt, factors, 16, stream);
        if (rc != WKV7_OK) return rc;
        return bwd(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, factors, 16, dy, dsT, dr, dw, dk, dv, da, db, ds0,
                   stream);
    }

    const Rows R(T, H, dtype);
    return run_blocks(B, n, static_cast<cudaStream_t>(stream), [&](int b0, int nb, cudaStream_t s) {
        int rc = fwd(nb, T, H, N, dtype, R.in(r, b0), R.in(w, b0), R.in(k, b0), R.in(v, b0), R.in(a, b0),
                     R.in(b, b0), R.at(s0, b0, R.state), R.at(y, b0, R.seq), R.at(sT, b0, R.state),
                     R.at(ckpt, b0, R.ck), R.at(factors, b0, R.fac), 16, s);
        if (rc != WKV7_OK) return rc;
        return bwd(nb, T, H, N, dtype, R.in(r, b0), R.in(w, b0), R.in(k, b0), R.in(v, b0), R.in(a, b0), R.in(b, b0),
                   R.at(ckpt, b0, R.ck), R.at(factors, b0, R.fac), 16, R.at(dy, b0, R.seq), R.at(dsT, b0, R.state),
                   R.at(dr, b0, R.seq), R.at(dw, b0, R.seq), R.at(dk, b0, R.seq), R.at(dv, b0, R.seq),
                   R.at(da, b0, R.seq), R.at(db, b0, R.seq), R.at(ds0, b0, R.state), s);
    });
}

}  // namespace

extern "C" {

int wkv7_forward_backward_blocks(int B, int T, int H, int nsplit) {
    if (B < 1 || H < 1 || T < 0 || nsplit < 0 || nsplit > kMaxSplit) return -1;
    return blocks_of(B, T, H, nsplit);
}

int wkv7_forward_backward(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w, const void *k,
                          const void *v, const void *a, const void *b, const float *s0, const float *dy,
                          const float *dsT, float *y, float *sT, float *ckpt, float *factors, float *dr, float *dw,
                          float *dk, float *dv, float *da, float *db, float *ds0, int nsplit, void *stream) {
    return step(wkv7_forward, wkv7_backward, false, B, T, H, N, dtype, r, w, k, v, a, b, s0, dy, dsT, y, sT, ckpt, factors,
                dr, dw, dk, dv, da, db, ds0, nsplit, stream);
}

int wkv7_forward_backward_fused(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w_pre,
                                const void *k, const void *v, const void *kk, const void *avec, const float *s0,
                                const float *dy, const float *dsT, float *y, float *sT, float *ckpt, float *factors,
                                float *dr, float *dw_pre, float *dk, float *dv, float *dkk, float *davec, float *ds0,
                                int nsplit, void *stream) {
    if (T > 0 && !factors) return wkv7::set_error(WKV7_EINVAL, "the fused producers' backward needs the factor cache");
    return step(wkv7_forward_fused, wkv7_backward_fused, true, B, T, H, N, dtype, r, w_pre, k, v, kk, avec, s0, dy, dsT,
                y, sT, ckpt, factors, dr, dw_pre, dk, dv, dkk, davec, ds0, nsplit, stream);
}

int wkv7_forward_backward_gn(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w,
                             const void *k, const void *v, const void *a, const void *b, const float *s0,
                             const float *do_, const float *dsT, const float *gn_w, const float *gn_b,
                             const float *r_k, float *y, float *o, float *sT, float *ckpt, float *factors, float *dr,
                             float *dw, float *dk, float *dv, float *da, float *db, float *ds0, float *dgn_w,
                             float *dgn_b, float *dr_k, float *workspace, int nsplit, void *stream) {
    if (check_nsplit(nsplit) != WKV7_OK) return WKV7_EINVAL;
    {   // every argument is checked before the first launch
        const void *req[17] = {r, w, k, v, a, b, do_, y, o, ckpt, factors, dr, dw, dk, dv, da, db};
        const char *rn[17] = {"r", "w", "k", "v", "a", "b", "do", "y", "o", "ckpt", "factors",
                              "dr", "dw", "dk", "dv", "da", "db"};
        // the epilogue's weights, parameter gradients and workspace (any T), then the rest
        const void *par[7] = {gn_w, gn_b, r_k, dgn_w, dgn_b, dr_k, workspace};
        const char *pn[7] = {"gn_w", "gn_b", "r_k", "dgn_w", "dgn_b", "dr_k", "workspace"};
        for (int i = 0; i < 7; ++i) {
            char msg[80];
            if (!par[i]) {
                snprintf(msg, sizeof msg, "%s is NULL", pn[i]);
                return wkv7::set_error(WKV7_EINVAL, msg);
            }
            if (reinterpret_cast<uintptr_t>(par[i]) & 15u) {
                snprintf(msg, sizeof msg, "%s is not 16-byte aligned", pn[i]);
                return wkv7::set_error(WKV7_EINVAL, msg);
            }
        }
        const void *opt[4] = {s0, dsT, sT, ds0};
        const char *on[4] = {"s0", "dsT", "sT", "ds0"};
        const int rc = wkv7::check_call(B, T, H, N, dtype, req, rn, 17, opt, on, 4);
        if (rc != WKV7_OK) return rc;
    }
    const int n = blocks_of(B, T, H, nsplit);
    if (n == 1) {  // one block: the two calls in order on the caller's stream
        int rc = wkv7_forward_gn(B, T, H, N, dtype, r, w, k, v, a, b, s0, gn_w, gn_b, r_k, y, o, sT, ckpt, factors, 16,
                                 stream);
        if (rc != WKV7_OK) return rc;
        return wkv7_backward_gn(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, factors, 16, y, do_, dsT, gn_w, r_k, dr, dw,
                                dk, dv, da, db, ds0, dgn_w, dgn_b, dr_k, workspace, stream);
    }
    // every block leaves its rows' per-(b, h) parameter-gradient sums in the
    // workspace; one reduction over all B rows follows once the blocks are joined
    const Rows R(T, H, dtype);
    const size_t wsrow = (size_t)H * 3 * WKV7_HEAD_SIZE;
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    int rc = run_blocks(B, n, caller, [&](int b0, int nb, cudaStream_t s) {
        int e = wkv7_forward_gn(nb, T, H, N, dtype, R.in(r, b0), R.in(w, b0), R.in(k, b0), R.in(v, b0), R.in(a, b0),
                                R.in(b, b0), R.at(s0, b0, R.state), gn_w, gn_b, r_k, R.at(y, b0, R.seq),
                                R.at(o, b0, R.seq), R.at(sT, b0, R.state), R.at(ckpt, b0, R.ck),
                                R.at(factors, b0, R.fac), 16, s);
        if (e != WKV7_OK) return e;
        return wkv7::backward_gn_partials(nb, T, H, N, dtype, R.in(r, b0), R.in(w, b0), R.in(k, b0), R.in(v, b0),
                                          R.in(a, b0), R.in(b, b0), R.at(ckpt, b0, R.ck), R.at(factors, b0, R.fac),
                                          R.at(y, b0, R.seq), R.at(do_, b0, R.seq), R.at(dsT, b0, R.state), gn_w, r_k,
                                          R.at(dr, b0, R.seq), R.at(dw, b0, R.seq), R.at(dk, b0, R.seq),
                                          R.at(dv, b0, R.seq), R.at(da, b0, R.seq), R.at(db, b0, R.seq),
                                          R.at(ds0, b0, R.state), workspace + (size_t)b0 * wsrow, s);
    });
    if (rc != WKV7_OK) return rc;
    const cudaError_t e = wkv7::launch_gn_param_reduce(B, H, workspace, dgn_w, dgn_b, dr_k, caller);
    return e == cudaSuccess ? WKV7_OK : cuda_fail(e, "parameter-gradient reduction launch");
}

}  // extern "C"
