// wkv7_forward_backward: one training step of the recurrence (the forward
// with checkpoints at stride 16 and the factor cache, then the backward) as
// concurrent sub-batches.
//
// Every (b, h) is independent in both directions, so the batch splits into
// nsplit contiguous row blocks, each running its forward and then its
// backward on a stream of its own: block 0 on the caller's stream, the others
// on streams of the library, forked from the caller's stream by an event and
// joined back into it, so the call stays stream-ordered for the caller.
// Using the caller's stream for one block keeps the library's own streams to
// nsplit - 1 (one for the default split): every stream more can share a
// hardware work queue with the caller's other streams, such as copy streams,
// and serialise work they meant to overlap.  A sub-batch's backward starts as soon as
// its own forward is done, while the other sub-batches' forward CTAs are
// still finishing; with one CTA per head the forward leaves a tail of
// unevenly loaded SMs and the backward a partly empty second wave, and the
// sub-batches fill each other's.
#include <cstdio>
#include <mutex>

#include "wkv7.h"
#include "wkv7_internal.cuh"

namespace {

constexpr int kMaxSplit = 4;
constexpr int kDefaultSplit = 2;
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
    if (nsplit < 0 || nsplit > kMaxSplit) {
        char msg[80];
        snprintf(msg, sizeof msg, "nsplit must be 0 (the default) .. %d (got %d)", kMaxSplit, nsplit);
        return wkv7::set_error(WKV7_EINVAL, msg);
    }
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
    int n = nsplit == 0 ? kDefaultSplit : nsplit;
    if (n > B) n = B;
    if (T == 0 || n == 1) {  // one block: the two calls in order on the caller's stream
        int rc = fwd(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, ckpt, factors, 16, stream);
        if (rc != WKV7_OK) return rc;
        return bwd(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, factors, 16, dy, dsT, dr, dw, dk, dv, da, db, ds0,
                   stream);
    }

    // element offsets of batch row b0 in each layout
    const size_t esize = dtype == WKV7_BF16 ? 2 : 4;
    const size_t seq = (size_t)T * H * WKV7_HEAD_SIZE;                              // [B][T][H][N] row
    const size_t state = (size_t)H * WKV7_HEAD_SIZE * WKV7_HEAD_SIZE;               // [B][H][N][N] row
    const size_t ck = state * (size_t)wkv7_ckpt_count(T, 16);                       // [B][H][nck][N][N] row
    const size_t fac = (size_t)H * (size_t)wkv7_factor_floats(T);                   // [B][H][factor floats] row
    auto in = [&](const void *p, int b0) {
        return static_cast<const void *>(static_cast<const char *>(p) + (size_t)b0 * seq * esize);
    };
    auto f32 = [](auto *p, int b0, size_t row) { return p ? p + (size_t)b0 * row : p; };

    std::lock_guard<std::mutex> lock(g_mu);
    Pool *pool = nullptr;
    int rc = pool_of_device(n, &pool);
    if (rc != WKV7_OK) return rc;
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(pool->fork, caller);
    if (e != cudaSuccess) return cuda_fail(e, "fork event");
    int joined = 1;  // library streams given work (1 .. joined - 1), joined back below even after an error
    for (int i = 0; i < n && rc == WKV7_OK; ++i) {
        const int b0 = (int)((long long)i * B / n), b1 = (int)((long long)(i + 1) * B / n), nb = b1 - b0;
        cudaStream_t s = i ? pool->s[i] : caller;
        if (i) {
            if ((e = cudaStreamWaitEvent(s, pool->fork, 0)) != cudaSuccess) {
                rc = cuda_fail(e, "fork wait");
                break;
            }
            joined = i + 1;
        }
        rc = fwd(nb, T, H, N, dtype, in(r, b0), in(w, b0), in(k, b0), in(v, b0), in(a, b0), in(b, b0),
                 f32(s0, b0, state), f32(y, b0, seq), f32(sT, b0, state), f32(ckpt, b0, ck), f32(factors, b0, fac),
                 16, s);
        if (rc != WKV7_OK) break;
        rc = bwd(nb, T, H, N, dtype, in(r, b0), in(w, b0), in(k, b0), in(v, b0), in(a, b0), in(b, b0),
                 f32(ckpt, b0, ck), f32(factors, b0, fac), 16, f32(dy, b0, seq), f32(dsT, b0, state),
                 f32(dr, b0, seq), f32(dw, b0, seq), f32(dk, b0, seq), f32(dv, b0, seq), f32(da, b0, seq),
                 f32(db, b0, seq), f32(ds0, b0, state), s);
    }
    for (int i = 1; i < joined; ++i) {
        const cudaError_t j1 = cudaEventRecord(pool->join[i], pool->s[i]);
        const cudaError_t j2 = j1 == cudaSuccess ? cudaStreamWaitEvent(caller, pool->join[i], 0) : j1;
        if (j2 != cudaSuccess && rc == WKV7_OK) rc = cuda_fail(j2, "join");
    }
    return rc;
}

}  // namespace

extern "C" {

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

}  // extern "C"
