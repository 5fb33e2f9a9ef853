// Sequence parallelism inside one GPU: each (b, h) sequence of T tokens is cut
// into nseg equal segments that run side by side as extra batch rows.
//
// Over a segment the recurrence is affine in its start state: with P_t =
// diag(w_t) + a_t b_t^T, S_end = S_start M + Z where M = P_1 ... P_L (the end
// state from S_start = I with v = 0) and Z is the end state from S_start = 0.
// The [B][T][H][N] inputs read as [B*nseg][T/nseg][H][N] make every segment
// an independent batch row, so:
//   forward: (1) all segments from S_start = I with v = 0  -> M,
//            (2) all segments from S_start = 0              -> Z,
//            (3) a scan over the segments of each head, S_{k+1} = S_k M_k + Z_k,
//            (4) all segments from their true start states -> y, checkpoints, factors;
//   backward (the adjoint of the same decomposition, with D_k = the gradient a
//   segment sends to its start state when nothing arrives at its end):
//            (1) all segments with no gradient at their end -> D,
//            (2) a reverse scan, G_{k-1} = D_k + G_k M_k^T from G_last = dsT,
//            (3) all segments with G_k arriving at their end -> the gradients.
// This is for few, long sequences (B*H small next to the GPU's CTA slots); it
// does about three times the forward work and twice the backward work.
#include <cstdio>

#include <cuda_runtime.h>

#include "wkv7.h"
#include "wkv7_internal.cuh"
#include "wkv7_mma.cuh"

namespace wkv7 {
// Runs work(i, stream, ctx) for i = 0 .. n - 1 side by side, piece 0 on
// `caller` and the others on the library's streams (wkv7_step.cu).
int run_side_by_side(int n, cudaStream_t caller, int (*work)(int, cudaStream_t, void *), void *ctx);
}  // namespace wkv7

namespace {
using wkv7::AFrag;
using wkv7::BFrag;
using wkv7::make_a;
using wkv7::make_b;
using wkv7::mma3;

constexpr int kN = 64;
constexpr int kPad = kN + 4;     // shared row stride (floats)
constexpr int kScanRows = 16;    // state rows per scan CTA
constexpr int kScanThreads = 128;

__device__ __forceinline__ size_t seg_off(int b, int k, int h, int nseg, int H) {
    return (((size_t)b * nseg + k) * H + h) * kN * kN;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}

// Per head (b, h): forward (kBack = false)
//   S_0 = init or 0;  for k = 0 .. nseg-1: out_k = S_k, S_{k+1} = C_k + S_k M_k;  fin = S_nseg
// backward (kBack = true)
//   G = init or 0;  for k = nseg-1 .. 0: out_k = G, G = C_k + G M_k^T;  fin = G
// (C = Z forward, D backward).  init / fin are [B][H][N][N] (either may be
// NULL); M, C, out are [B][nseg][H][N][N].
// Row i of the next state depends on row i of the current one only, so a
// head's 64 rows run as 4 CTAs of 16 (blockIdx.y); warp w of a CTA owns
// columns 16w .. 16w + 15.  Each step's 16 x 64 x 64 product runs on the
// tensor cores with split operands (bf16x3, fp32 accumulation); the next
// step's M arrives by cp.async into the other buffer during the products.
template <bool kBack>
__global__ void __launch_bounds__(kScanThreads) wkv7_segment_scan_kernel(int H, int nseg, const float *__restrict__ M,
                                                                         const float *__restrict__ Cadd,
                                                                         const float *__restrict__ init,
                                                                         float *__restrict__ out,
                                                                         float *__restrict__ fin) {
    __shared__ __align__(16) float Ms[2][kN * kPad];         // M_k, double-buffered
    __shared__ __align__(16) float Ss[2][kScanRows * kPad];  // this CTA's rows of the current state
    const int bh = blockIdx.x, b = bh / H, h = bh % H, row0 = kScanRows * blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q = lane & 3;
    const size_t head = (size_t)bh * kN * kN;
    auto seg = [&](int step) { return kBack ? nseg - 1 - step : step; };
    auto stage_m = [&](int step, float *dst) {  // 1024 16-byte pieces, 8 per thread
        const float *src = M + seg_off(b, seg(step), h, nseg, H);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int e = tid + kScanThreads * m, row = e >> 4, c4 = (e & 15) * 4;
            cp_async16(dst + row * kPad + c4, src + row * kN + c4);
        }
        cp_async_commit();
    };
    // every step's operands are independent of the scan: ask L2 for all of them now (each
    // of a head's four CTAs a quarter of the M_k, and its own rows of every C_k), so that
    // the steps' copies do not wait on DRAM
    for (int k = tid; k < nseg; k += kScanThreads) {
        const size_t o = seg_off(b, k, h, nseg, H);
        if ((k & 3) == (int)blockIdx.y) prefetch_l2(M + o, kN * kN * 4);
        prefetch_l2(Cadd + o + (size_t)row0 * kN, kScanRows * kN * 4);
    }
    stage_m(0, Ms[0]);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int e = tid + kScanThreads * m, r = e >> 4, c4 = (e & 15) * 4;
        const float4 x = init ? *reinterpret_cast<const float4 *>(init + head + (row0 + r) * kN + c4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Ss[0] + r * kPad + c4) = x;
    }
    auto load_c = [&](int step, float (*c)[4]) {  // the additive term at this lane's positions
        const float *cb = Cadd + seg_off(b, seg(step), h, nseg, H) + (size_t)(row0 + g) * kN + 16 * warp + 2 * q;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float2 x = *reinterpret_cast<const float2 *>(cb + 8 * u);
            const float2 z = *reinterpret_cast<const float2 *>(cb + 8 * u + 8 * kN);
            c[u][0] = x.x; c[u][1] = x.y; c[u][2] = z.x; c[u][3] = z.y;
        }
    };
    float acc[2][4];  // the next state at rows row0 + g (+8), columns 16 warp + 8u + 2q (+1)
    float cn[2][4];   // the next step's additive term, loaded a step ahead
    load_c(0, cn);
    for (int step = 0; step < nseg; ++step) {
        const int cur = step & 1;
        const size_t o = seg_off(b, seg(step), h, nseg, H);
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[u][e] = cn[u][e];
        cp_async_wait_all();
        __syncthreads();  // M_k and the current rows are visible; step - 1 no longer reads the other buffers
        if (step + 1 < nseg) {
            stage_m(step + 1, Ms[cur ^ 1]);
            load_c(step + 1, cn);
        }
        const float *Mk = Ms[cur], *Sk = Ss[cur];
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // out_k = the current rows
            const int e = tid + kScanThreads * m, r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4 *>(out + o + (row0 + r) * kN + c4) = *reinterpret_cast<const float4 *>(Sk + r * kPad + c4);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float *a = Sk + g * kPad + 16 * kk + 2 * q;
            auto ld2 = [](const float *x) { return *reinterpret_cast<const float2 *>(x); };
            const AFrag af = make_a(ld2(a), ld2(a + 8 * kPad), ld2(a + 8), ld2(a + 8 * kPad + 8));
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int n = 16 * warp + 8 * u + g, k0 = 16 * kk + 2 * q;
                BFrag bf;
                if (kBack)  // B[k][n] = M[n][k]
                    bf = make_b(ld2(Mk + n * kPad + k0), ld2(Mk + n * kPad + k0 + 8));
                else        // B[k][n] = M[k][n]
                    bf = make_b(make_float2(Mk[k0 * kPad + n], Mk[(k0 + 1) * kPad + n]),
                                make_float2(Mk[(k0 + 8) * kPad + n], Mk[(k0 + 9) * kPad + n]));
                mma3(acc[u], af, bf);
            }
        }
        float *Sn = Ss[cur ^ 1];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c = 16 * warp + 8 * u + 2 * q;
            *reinterpret_cast<float2 *>(Sn + g * kPad + c) = make_float2(acc[u][0], acc[u][1]);
            *reinterpret_cast<float2 *>(Sn + (g + 8) * kPad + c) = make_float2(acc[u][2], acc[u][3]);
        }
    }
    if (fin) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float *fp = fin + head + (size_t)(row0 + g) * kN + 16 * warp + 8 * u + 2 * q;
            *reinterpret_cast<float2 *>(fp) = make_float2(acc[u][0], acc[u][1]);
            *reinterpret_cast<float2 *>(fp + 8 * kN) = make_float2(acc[u][2], acc[u][3]);
        }
    }
}

// n identity matrices [n][N][N]
__global__ void wkv7_identity_kernel(float *dst, size_t n) {
    const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n * kN * kN) return;
    const int rc = (int)(e % (kN * kN));
    dst[e] = (rc / kN == rc % kN) ? 1.f : 0.f;
}

struct Workspace {
    float *M, *Z, *starts, *D, *G, *ident, *ckpt, *fac;
};

long long state_floats(int B, int H, int nseg) { return (long long)B * nseg * H * kN * kN; }

Workspace carve(float *ws, int B, int T, int H, int nseg) {
    const long long s = state_floats(B, H, nseg);
    const int tseg = T / nseg;
    Workspace w;
    w.M = ws;
    w.Z = w.M + s;
    w.starts = w.Z + s;
    w.D = w.starts + s;
    w.G = w.D + s;
    w.ident = w.G + s;
    w.ckpt = w.ident + s;
    w.fac = w.ckpt + (long long)B * nseg * H * wkv7_ckpt_count(tseg, 16) * kN * kN;
    return w;
}

int check_split(int B, int T, int H, int nseg, const float *ws) {
    if (B < 1 || H < 1 || T < 0) return wkv7::set_error(WKV7_EINVAL, "B, H must be >= 1 and T >= 0");
    if (nseg < 1) return wkv7::set_error(WKV7_EINVAL, "nseg must be >= 1");
    if (T % (16 * nseg) != 0) return wkv7::set_error(WKV7_EINVAL, "T must be a multiple of 16 * nseg");
    if ((long long)B * nseg * H > 0x7fffffffLL) return wkv7::set_error(WKV7_EINVAL, "B * nseg * H too large");
    if (T > 0 && !ws) return wkv7::set_error(WKV7_EINVAL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 15u) return wkv7::set_error(WKV7_EINVAL, "workspace is not 16-byte aligned");
    return WKV7_OK;
}

int cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return WKV7_OK;
    char msg[160];
    snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return wkv7::set_error(WKV7_ECUDA, msg);
}

}  // namespace

extern "C" {

long long wkv7_timesplit_workspace_floats(int B, int T, int H, int nseg) {
    if (B < 1 || H < 1 || T < 0 || nseg < 1 || T % (16 * nseg) != 0) return -1;
    const int tseg = T / nseg;
    const long long s = state_floats(B, H, nseg);
    return 6 * s + (long long)B * nseg * H * wkv7_ckpt_count(tseg, 16) * kN * kN +
           (long long)B * nseg * H * wkv7_factor_floats(tseg);
}

int wkv7_segment_scan(int B, int H, int nseg, const float *M, const float *C, const float *init, float *out,
                      float *fin, int backward, void *stream) {
    if (B < 1 || H < 1 || nseg < 1) return wkv7::set_error(WKV7_EINVAL, "B, H and nseg must be >= 1");
    if ((long long)B * H > 0x7fffffffLL) return wkv7::set_error(WKV7_EINVAL, "B * H too large");
    const void *ptrs[5] = {M, C, init, out, fin};
    const char *names[5] = {"M", "C", "init", "out", "fin"};
    for (int i = 0; i < 5; ++i) {
        if (!ptrs[i] && i < 2) return wkv7::set_error(WKV7_EINVAL, i ? "C is NULL" : "M is NULL");
        if (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) {
            char msg[64];
            snprintf(msg, sizeof msg, "%s is not 16-byte aligned", names[i]);
            return wkv7::set_error(WKV7_EINVAL, msg);
        }
    }
    if (!out) return wkv7::set_error(WKV7_EINVAL, "out is NULL");
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
        minor != 3) {
        cudaGetLastError();
        return wkv7::set_error(WKV7_EUNSUPPORTED, "this library needs an sm_103a device");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(B * H, kN / kScanRows);
    if (backward)
        wkv7_segment_scan_kernel<true><<<grid, kScanThreads, 0, st>>>(H, nseg, M, C, init, out, fin);
    else
        wkv7_segment_scan_kernel<false><<<grid, kScanThreads, 0, st>>>(H, nseg, M, C, init, out, fin);
    return cuda_status(cudaGetLastError(), "segment scan launch");
}

int wkv7_forward_timesplit(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w,
                           const void *k, const void *v, const void *a, const void *b, const float *s0, float *y,
                           float *sT, int nseg, float *workspace, void *stream) {
    int rc = check_split(B, T, H, nseg, workspace);
    if (rc != WKV7_OK) return rc;
    {   // every argument is checked before the first launch or memset
        const void *req[7] = {r, w, k, v, a, b, y};
        const char *rn[7] = {"r", "w", "k", "v", "a", "b", "y"};
        const void *opt[2] = {s0, sT};
        const char *on[2] = {"s0", "sT"};
        rc = wkv7::check_call(B, T, H, N, dtype, req, rn, 7, opt, on, 2);
        if (rc != WKV7_OK) return rc;
    }
    if (T == 0) return wkv7_forward(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, nullptr, nullptr, 16, stream);
    const int bs = B * nseg, tseg = T / nseg;
    const Workspace ws = carve(workspace, B, T, H, nseg);
    if (nseg == 1)  // one segment: the plain call, keeping its checkpoints and factors for the backward
        return wkv7_forward(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, ws.ckpt, ws.fac, 16, stream);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long s = state_floats(B, H, nseg);
    const size_t nmat = (size_t)bs * H;
    wkv7_identity_kernel<<<(unsigned)((s + 255) / 256), 256, 0, st>>>(ws.ident, nmat);
    if ((rc = cuda_status(cudaGetLastError(), "identity launch")) != WKV7_OK) return rc;
    // (1) M: every segment from I with v = 0 -- the segment pass that reads only w, a, b
    // and forms no V product and no y; (2) Z: every segment from 0 (end state only, no y).
    // The two are independent and, with B*H small, each fills only part of the GPU:
    // they run side by side, M on a stream of the library's forked from this one.
    struct Passes {
        int bs, tseg, H, dtype;
        const void *w, *k, *v, *a, *b;
        const float *ident;
        float *M, *Z;
    } ps{bs, tseg, H, dtype, w, k, v, a, b, ws.ident, ws.M, ws.Z};
    rc = wkv7::run_side_by_side(2, st, [](int i, cudaStream_t s, void *c) -> int {
        const Passes &x = *static_cast<const Passes *>(c);
        return i ? wkv7::forward_state(x.bs, x.tseg, x.H, x.dtype, x.w, x.k, x.v, x.a, x.b, x.ident, x.M, 2, s)
                 : wkv7::forward_state(x.bs, x.tseg, x.H, x.dtype, x.w, x.k, x.v, x.a, x.b, nullptr, x.Z, 1, s);
    }, &ps);
    if (rc) return rc;
    // (3) segment start states, and the final state
    wkv7_segment_scan_kernel<false><<<dim3(B * H, kN / kScanRows), kScanThreads, 0, st>>>(H, nseg, ws.M, ws.Z, s0,
                                                                                           ws.starts, sT);
    if ((rc = cuda_status(cudaGetLastError(), "segment scan launch")) != WKV7_OK) return rc;
    // (4) every segment from its start state; checkpoints and factors for the backward
    return wkv7_forward(bs, tseg, H, N, dtype, r, w, k, v, a, b, ws.starts, y, nullptr, ws.ckpt, ws.fac, 16, stream);
}

int wkv7_backward_timesplit(int B, int T, int H, int N, wkv7_dtype dtype, const void *r, const void *w,
                            const void *k, const void *v, const void *a, const void *b, const float *dy,
                            const float *dsT, float *dr, float *dw, float *dk, float *dv, float *da, float *db,
                            float *ds0, int nseg, float *workspace, void *stream) {
    int rc = check_split(B, T, H, nseg, workspace);
    if (rc != WKV7_OK) return rc;
    {   // every argument is checked before the first launch
        const void *req[13] = {r, w, k, v, a, b, dy, dr, dw, dk, dv, da, db};
        const char *rn[13] = {"r", "w", "k", "v", "a", "b", "dy", "dr", "dw", "dk", "dv", "da", "db"};
        const void *opt[2] = {dsT, ds0};
        const char *on[2] = {"dsT", "ds0"};
        rc = wkv7::check_call(B, T, H, N, dtype, req, rn, 13, opt, on, 2);
        if (rc != WKV7_OK) return rc;
    }
    if (T == 0) return wkv7_backward(B, 0, H, N, dtype, r, w, k, v, a, b, nullptr, nullptr, 16, dy, dsT, dr, dw, dk,
                                     dv, da, db, ds0, stream);
    const int bs = B * nseg, tseg = T / nseg;
    const Workspace ws = carve(workspace, B, T, H, nseg);
    if (nseg == 1)
        return wkv7_backward(B, T, H, N, dtype, r, w, k, v, a, b, ws.ckpt, ws.fac, 16, dy, dsT, dr, dw, dk, dv, da, db,
                             ds0, stream);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // (1) no gradient arriving at the segment ends: D = what each segment sends to its start
    // (the state gradient alone, from the factors the forward kept)
    if ((rc = wkv7::backward_state(bs, tseg, H, dtype, r, w, a, b, ws.fac, dy, nullptr, ws.D, st)))
        return rc;
    // (2) the gradient arriving at every segment's end, and ds0
    wkv7_segment_scan_kernel<true><<<dim3(B * H, kN / kScanRows), kScanThreads, 0, st>>>(H, nseg, ws.M, ws.D, dsT,
                                                                                          ws.G, ds0);
    if ((rc = cuda_status(cudaGetLastError(), "segment scan launch")) != WKV7_OK) return rc;
    // (3) the gradients, each segment with its arriving gradient (its own ds0 is not needed)
    return wkv7_backward(bs, tseg, H, N, dtype, r, w, k, v, a, b, ws.ckpt, ws.fac, 16, dy, ws.G, dr, dw, dk, dv, da,
                         db, ws.starts, stream);
}

}  // extern "C"
