// Per-token WKV7 kernels: sequence forward, reverse-time backward and the
// single-token decode step.
//
// The recurrence, per (b,h), state S[i][j] (i value row, j key column):
//   sa_t = S_{t-1} a_t ;  S_t = S_{t-1} diag(w_t) + sa_t b_t^T + v_t k_t^T ;
//   y_t  = S_t r_t.
// Layouts follow the "Foundry/cuda_kernels/timemix.cu" page (file header):
// token vectors [B][T][H][N], state [B][H][N][N]; the adjoint follows the
// "WKV kernel backward" block of accumulate_token_step_gradients on the
// "infotheory/backends/rwkvzip/rwkv7/model.rs" page, and the backward replays
// each checkpoint interval forward the way online_train_segment_tbptt on that
// page replays its chunks.
//
// Thread layout (all three kernels): one CTA of 256 threads per (b,h).
// Thread (rg, cg), rg, cg in [0,16), holds the 4x4 block of S with rows
// 4rg..4rg+3 and columns 4cg..4cg+3 in registers.  The 16 column groups of a
// row group are the 16 lanes of one half warp, so row reductions (S a, S r,
// G b, G k) are half-warp shuffles; column reductions (the key-side
// gradients) finish across the eight warps through shared memory.  Every
// reduction has a fixed order: results are bit-reproducible.
#include "wkv7_internal.cuh"

namespace wkv7 {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 16;  // tokens per staged forward chunk
constexpr int kWin = 8;     // tokens per backward window (states kept in smem)
constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ void to4(const float4 q, float o[4]) { o[0] = q.x; o[1] = q.y; o[2] = q.z; o[3] = q.w; }

// Sum 4 per-row partials over the 16 lanes of a half warp; every lane gets
// all 4 row sums.  Transposed butterfly: 9 shuffles instead of 16.  The
// result is identical on every lane (IEEE addition is commutative).
__device__ __forceinline__ void allreduce_rows(float p[4], int lane) {
    const bool hi = lane & 8;
    const float s0 = hi ? p[0] : p[2], s1 = hi ? p[1] : p[3];
    float k0 = hi ? p[2] : p[0], k1 = hi ? p[3] : p[1];
    k0 += __shfl_xor_sync(kFull, s0, 8);
    k1 += __shfl_xor_sync(kFull, s1, 8);
    const bool h4 = lane & 4;
    const float snd = h4 ? k0 : k1;
    float kp = h4 ? k1 : k0;
    kp += __shfl_xor_sync(kFull, snd, 4);
    kp += __shfl_xor_sync(kFull, kp, 2);
    kp += __shfl_xor_sync(kFull, kp, 1);
    const int base = lane & 16;
    p[0] = __shfl_sync(kFull, kp, base | 0);
    p[1] = __shfl_sync(kFull, kp, base | 4);
    p[2] = __shfl_sync(kFull, kp, base | 8);
    p[3] = __shfl_sync(kFull, kp, base | 12);
}

// Same sum without the final broadcast: returns the full sum of row
// m = 2*bit3(lane) + bit2(lane) of the lane's row group.
__device__ __forceinline__ float reduce_rows(const float p[4], int lane) {
    const bool hi = lane & 8;
    const float s0 = hi ? p[0] : p[2], s1 = hi ? p[1] : p[3];
    float k0 = hi ? p[2] : p[0], k1 = hi ? p[3] : p[1];
    k0 += __shfl_xor_sync(kFull, s0, 8);
    k1 += __shfl_xor_sync(kFull, s1, 8);
    const bool h4 = lane & 4;
    const float snd = h4 ? k0 : k1;
    float kp = h4 ? k1 : k0;
    kp += __shfl_xor_sync(kFull, snd, 4);
    kp += __shfl_xor_sync(kFull, kp, 2);
    kp += __shfl_xor_sync(kFull, kp, 1);
    return kp;
}
__device__ __forceinline__ int reduced_row(int lane) { return ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1); }

// One recurrence step on the thread's 4x4 block.  Explicit _rn intrinsics
// fix the instruction sequence, so every kernel that calls this produces
// bit-identical states from identical inputs (the backward's replay matches
// the forward's checkpoints).  On return sa[] holds S_{t-1} a_t for the 4 rows.
__device__ __forceinline__ void step(float s[4][4], const float w[4], const float k[4],
                                     const float a[4], const float b[4], const float v[4],
                                     float sa[4], int lane) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float acc = __fmul_rn(s[m][0], a[0]);
        acc = __fmaf_rn(s[m][1], a[1], acc);
        acc = __fmaf_rn(s[m][2], a[2], acc);
        sa[m] = __fmaf_rn(s[m][3], a[3], acc);
    }
    allreduce_rows(sa, lane);
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n)
            s[m][n] = __fmaf_rn(s[m][n], w[n], __fmaf_rn(sa[m], b[n], __fmul_rn(v[m], k[n])));
}

__device__ __forceinline__ void dot_rows(const float s[4][4], const float x[4], float p[4]) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float acc = __fmul_rn(s[m][0], x[0]);
        acc = __fmaf_rn(s[m][1], x[1], acc);
        acc = __fmaf_rn(s[m][2], x[2], acc);
        p[m] = __fmaf_rn(s[m][3], x[3], acc);
    }
}

__device__ __forceinline__ void load_block(float s[4][4], const float *src, int rg, int cg) {
#pragma unroll
    for (int m = 0; m < 4; ++m) to4(*reinterpret_cast<const float4 *>(src + (rg * 4 + m) * kN + cg * 4), s[m]);
}
__device__ __forceinline__ void store_block(const float s[4][4], float *dst, int rg, int cg) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
        *reinterpret_cast<float4 *>(dst + (rg * 4 + m) * kN + cg * 4) = make_float4(s[m][0], s[m][1], s[m][2], s[m][3]);
}

// ---- staging: token vectors -> shared memory
// Element type E of r,w,k,v,a,b as stored in global memory.
template <typename E>
struct Stage;

template <>
struct Stage<float> {
    // raw smem block [vec][tok][64] floats; read 4 contiguous floats at (vec,tok,n)
    static __device__ __forceinline__ void read4(const void *raw, int ntok, int vec, int u, int n, float o[4]) {
        to4(*reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(raw) + ((size_t)vec * ntok + u) * kN + n), o);
    }
};
template <>
struct Stage<__nv_bfloat16> {
    static __device__ __forceinline__ void read4(const void *raw, int ntok, int vec, int u, int n, float o[4]) {
        const uint2 q = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(raw) + ((size_t)vec * ntok + u) * kN + n);
        o[0] = bf16_lo(q.x); o[1] = bf16_hi(q.x); o[2] = bf16_lo(q.y); o[3] = bf16_hi(q.y);
    }
};

// Issue cp.async copies of NV vectors (src[0..NV-1]) for tokens
// [t0, t0+ntok) into raw smem [NV][ntok][64] of element E; tokens >= nvalid
// are zero-filled.  `base` is the element offset of (b, t0, h, 0) and
// `tstride` = H*N the element stride between tokens.
template <typename E, int NV>
__device__ __forceinline__ void stage_async(E *raw, const E *const (&src)[NV], size_t base, size_t tstride,
                                            int ntok, int nvalid) {
    constexpr int P = 16 / sizeof(E);  // elements per 16-byte copy
    const int per_tok = kN / P;
    const int per_vec = ntok * per_tok;
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
        for (int e = threadIdx.x; e < per_vec; e += kThreads) {
            const int u = e / per_tok, n = (e % per_tok) * P;
            const bool ok = u < nvalid;
            const E *g = ok ? src[vv] + base + (size_t)u * tstride + n : src[vv];
            cp_async16(raw + ((size_t)vv * ntok + u) * kN + n, g, ok ? 16 : 0);
        }
    }
}

// ------------------------------------------------------------------ forward

// Vector order in the staged block.
enum { VR = 0, VW = 1, VK = 2, VV = 3, VA = 4, VB = 5 };

template <typename E>
__global__ void __launch_bounds__(kThreads) wkv7_fwd_plain_kernel(SeqArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);                                   // [2][6][kChunk][64]
    float *ys = reinterpret_cast<float *>(smem + 2 * 6 * kChunk * kN * sizeof(E));  // [2][kChunk][64]

    const int bh = blockIdx.x;
    const int bi = bh / p.H, h = bh % p.H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cg = lane & 15, rg = warp * 2 + (lane >> 4);
    const size_t tstride = (size_t)p.H * kN;
    const size_t base0 = ((size_t)bi * p.T * p.H + h) * kN;  // (b, t=0, h, 0)
    const size_t sbase = (size_t)bh * kN * kN;

    float s[4][4];
    if (p.s0) load_block(s, p.s0 + sbase, rg, cg);
    else {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) s[m][n] = 0.f;
    }

    const E *const src[6] = {static_cast<const E *>(p.r), static_cast<const E *>(p.w), static_cast<const E *>(p.k),
                             static_cast<const E *>(p.v), static_cast<const E *>(p.a), static_cast<const E *>(p.b)};
    const int nchunks = (p.T + kChunk - 1) / kChunk;
    const size_t rawsz = (size_t)6 * kChunk * kN;

    if (nchunks > 0) stage_async<E, 6>(raw, src, base0, tstride, kChunk, min(kChunk, p.T));
    cp_async_commit();

    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kChunk;
        const int nt = min(kChunk, p.T - t0);
        if (c + 1 < nchunks)
            stage_async<E, 6>(raw + ((c + 1) & 1) * rawsz, src, base0 + (size_t)(t0 + kChunk) * tstride, tstride,
                              kChunk, min(kChunk, p.T - t0 - kChunk));
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const E *cur = raw + (c & 1) * rawsz;
        float *ycur = ys + (c & 1) * kChunk * kN;
        for (int u = 0; u < nt; ++u) {
            const int t = t0 + u;
            if (p.ckpt && t % p.L == 0)
                store_block(s, p.ckpt + ((size_t)bh * p.nck + t / p.L) * kN * kN, rg, cg);
            float w[4], k[4], a[4], b[4], v[4], r[4], sa[4], q[4];
            Stage<E>::read4(cur, kChunk, VW, u, cg * 4, w);
            Stage<E>::read4(cur, kChunk, VK, u, cg * 4, k);
            Stage<E>::read4(cur, kChunk, VA, u, cg * 4, a);
            Stage<E>::read4(cur, kChunk, VB, u, cg * 4, b);
            Stage<E>::read4(cur, kChunk, VV, u, rg * 4, v);
            step(s, w, k, a, b, v, sa, lane);
            Stage<E>::read4(cur, kChunk, VR, u, cg * 4, r);
            dot_rows(s, r, q);
            const float yv = reduce_rows(q, lane);
            if ((lane & 3) == 0) ycur[u * kN + rg * 4 + reduced_row(lane)] = yv;
        }
        __syncthreads();
        // write this chunk's y: nt tokens x 64 floats, one float4 per thread per 16 floats
        for (int e = threadIdx.x; e < nt * (kN / 4); e += kThreads) {
            const int u = e / (kN / 4), n = (e % (kN / 4)) * 4;
            *reinterpret_cast<float4 *>(p.y + base0 + (size_t)(t0 + u) * tstride + n) =
                *reinterpret_cast<const float4 *>(ycur + u * kN + n);
        }
    }
    cp_async_wait<0>();
    if (p.sT) store_block(s, p.sT + sbase, rg, cg);
}

// ----------------------------------------------------------------- backward
//
// For each checkpoint interval c (last to first), windows of kWin tokens are
// processed last to first.  For a window [ws, we): the state is reloaded
// from ckpt[c] and replayed forward to token ws, then replayed through the
// window keeping every state S_{t-1}, S_t in shared memory (each thread
// keeps its own 4x4 block, so this part needs no synchronisation) and sa_t.
// The reverse sweep then carries G = dL/dS_t:
//   G += dy_t r_t^T ; dr_t = S_t^T dy_t ; dv_t = G k_t ; dsa = G b_t ;
//   dk_t = G^T v_t ; db_t = G^T sa_t ; dw_t = colsum(G o S_{t-1}) ;
//   da_t = S_{t-1}^T dsa ; G <- G diag(w_t) + dsa a_t^T.

enum { BR = 0, BW = 1, BK = 2, BV = 3, BA = 4, BB = 5 };  // staged input vectors
enum { GR = 0, GK = 1, GB = 2, GW = 3, GA = 4, GV = 5 };  // staged gradient vectors

struct BwdSmem {
    static constexpr size_t hist = (size_t)(kWin + 1) * kN * kN * sizeof(float);
    static constexpr size_t dyb = (size_t)kWin * kN * sizeof(float);
    static constexpr size_t sab = (size_t)kWin * kN * sizeof(float);
    static constexpr size_t red = (size_t)2 * 8 * 10 * 32 * sizeof(float);
    static constexpr size_t grad = (size_t)6 * kWin * kN * sizeof(float);
    template <typename E>
    static constexpr size_t raw() { return (size_t)6 * kWin * kN * sizeof(E); }
    template <typename E>
    static constexpr size_t total() { return hist + dyb + sab + red + grad + raw<E>(); }
};

template <typename E>
__global__ void __launch_bounds__(kThreads, 1) wkv7_bwd_plain_kernel(SeqArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *hist = reinterpret_cast<float *>(smem);                     // [kWin+1][64][64]
    float *dys = reinterpret_cast<float *>(smem + BwdSmem::hist);     // [kWin][64]
    float *sas = dys + kWin * kN;                                      // [kWin][64]
    float *red = sas + kWin * kN;                                      // [2][8 warps*10][32]
    float *gst = red + 2 * 8 * 10 * 32;                                // [6][kWin][64]
    E *raw = reinterpret_cast<E *>(gst + 6 * kWin * kN);               // [6][kWin][64]

    const int bh = blockIdx.x;
    const int bi = bh / p.H, h = bh % p.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane & 15, rg = warp * 2 + (lane >> 4);
    const int half = lane >> 4;
    const size_t tstride = (size_t)p.H * kN;
    const size_t base0 = ((size_t)bi * p.T * p.H + h) * kN;
    const size_t sbase = (size_t)bh * kN * kN;
    const E *const src[6] = {static_cast<const E *>(p.r), static_cast<const E *>(p.w), static_cast<const E *>(p.k),
                             static_cast<const E *>(p.v), static_cast<const E *>(p.a), static_cast<const E *>(p.b)};
    const float *const dsrc[1] = {p.dy};
    float *const gout[6] = {p.dr, p.dk, p.db, p.dw, p.da, p.dv};

    float G[4][4];
    if (p.dsT) load_block(G, p.dsT + sbase, rg, cg);
    else {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) G[m][n] = 0.f;
    }
    float *myhist = hist;  // thread-private 4x4 blocks live at their natural (row, col) spots

    for (int c = p.nck - 1; c >= 0; --c) {
        const int t0 = c * p.L;
        const int t1 = min(p.T, t0 + p.L);
        const int nwin = (t1 - t0 + kWin - 1) / kWin;
        for (int wi = nwin - 1; wi >= 0; --wi) {
            const int ws = t0 + wi * kWin;
            const int nt = min(kWin, t1 - ws);
            // ---- replay from the checkpoint to token ws
            float s[4][4];
            load_block(s, p.ckpt_in + ((size_t)bh * p.nck + c) * kN * kN, rg, cg);
            for (int rs = t0; rs < ws; rs += kWin) {
                __syncthreads();
                stage_async<E, 6>(raw, src, base0 + (size_t)rs * tstride, tstride, kWin, kWin);
                cp_async_commit();
                cp_async_wait<0>();
                __syncthreads();
                for (int u = 0; u < kWin; ++u) {
                    float w[4], k[4], a[4], b[4], v[4], sa[4];
                    Stage<E>::read4(raw, kWin, BW, u, cg * 4, w);
                    Stage<E>::read4(raw, kWin, BK, u, cg * 4, k);
                    Stage<E>::read4(raw, kWin, BA, u, cg * 4, a);
                    Stage<E>::read4(raw, kWin, BB, u, cg * 4, b);
                    Stage<E>::read4(raw, kWin, BV, u, rg * 4, v);
                    step(s, w, k, a, b, v, sa, lane);
                }
            }
            // ---- stage the window's inputs and dy
            __syncthreads();
            stage_async<E, 6>(raw, src, base0 + (size_t)ws * tstride, tstride, kWin, nt);
            stage_async<float, 1>(dys, dsrc, base0 + (size_t)ws * tstride, tstride, kWin, nt);
            cp_async_commit();
            cp_async_wait<0>();
            __syncthreads();
            // ---- replay through the window, keeping states and sa
            store_block(s, myhist, rg, cg);
            for (int u = 0; u < nt; ++u) {
                float w[4], k[4], a[4], b[4], v[4], sa[4];
                Stage<E>::read4(raw, kWin, BW, u, cg * 4, w);
                Stage<E>::read4(raw, kWin, BK, u, cg * 4, k);
                Stage<E>::read4(raw, kWin, BA, u, cg * 4, a);
                Stage<E>::read4(raw, kWin, BB, u, cg * 4, b);
                Stage<E>::read4(raw, kWin, BV, u, rg * 4, v);
                step(s, w, k, a, b, v, sa, lane);
                store_block(s, myhist + (size_t)(u + 1) * kN * kN, rg, cg);
                if (cg == 0) *reinterpret_cast<float4 *>(sas + u * kN + rg * 4) = make_float4(sa[0], sa[1], sa[2], sa[3]);
            }
            __syncthreads();
            // ---- reverse sweep over the window
            for (int u = nt - 1; u >= 0; --u) {
                float r[4], w[4], k[4], a[4], b[4], v[4], dy[4], sa[4];
                Stage<E>::read4(raw, kWin, BR, u, cg * 4, r);
                Stage<E>::read4(raw, kWin, BW, u, cg * 4, w);
                Stage<E>::read4(raw, kWin, BK, u, cg * 4, k);
                Stage<E>::read4(raw, kWin, BA, u, cg * 4, a);
                Stage<E>::read4(raw, kWin, BB, u, cg * 4, b);
                Stage<E>::read4(raw, kWin, BV, u, rg * 4, v);
                to4(*reinterpret_cast<const float4 *>(dys + u * kN + rg * 4), dy);
                to4(*reinterpret_cast<const float4 *>(sas + u * kN + rg * 4), sa);
                float sn[4][4], sp[4][4];
                load_block(sn, myhist + (size_t)(u + 1) * kN * kN, rg, cg);
                load_block(sp, myhist + (size_t)u * kN * kN, rg, cg);

#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n) G[m][n] = __fmaf_rn(dy[m], r[n], G[m][n]);

                float pv[4], pd[4];
                dot_rows(G, k, pv);
                dot_rows(G, b, pd);
                const float dvv = reduce_rows(pv, lane);
                allreduce_rows(pd, lane);  // pd[m] = dsa for row 4rg+m

                // column partials over the thread's 4 rows: dr, dk, db, dw, da
                float P[20];
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    float xr = __fmul_rn(sn[0][n], dy[0]);
                    float xk = __fmul_rn(G[0][n], v[0]);
                    float xb = __fmul_rn(G[0][n], sa[0]);
                    float xw = __fmul_rn(G[0][n], sp[0][n]);
                    float xa = __fmul_rn(sp[0][n], pd[0]);
#pragma unroll
                    for (int m = 1; m < 4; ++m) {
                        xr = __fmaf_rn(sn[m][n], dy[m], xr);
                        xk = __fmaf_rn(G[m][n], v[m], xk);
                        xb = __fmaf_rn(G[m][n], sa[m], xb);
                        xw = __fmaf_rn(G[m][n], sp[m][n], xw);
                        xa = __fmaf_rn(sp[m][n], pd[m], xa);
                    }
                    P[GR * 4 + n] = xr; P[GK * 4 + n] = xk; P[GB * 4 + n] = xb; P[GW * 4 + n] = xw; P[GA * 4 + n] = xa;
                }
                // carried gradient to the previous state
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n) G[m][n] = __fmaf_rn(G[m][n], w[n], __fmul_rn(pd[m], a[n]));

                // column reduction: half-warp pair (xor 16), then the 8 warps via smem
                float *rb = red + (u & 1) * (8 * 10 * 32);
#pragma unroll
                for (int i = 0; i < 10; ++i) {
                    const float keep = half ? P[10 + i] : P[i];
                    const float send = half ? P[i] : P[10 + i];
                    rb[(warp * 10 + i) * 32 + lane] = keep + __shfl_xor_sync(kFull, send, 16);
                }
                if ((lane & 3) == 0) gst[(GV * kWin + u) * kN + rg * 4 + reduced_row(lane)] = dvv;
                __syncthreads();
                for (int o = tid; o < 5 * kN; o += kThreads) {
                    const int g = o / kN, j = o % kN;
                    const int idx = g * 4 + (j & 3);
                    const int hh = idx >= 10 ? 1 : 0;
                    const int slot = idx - hh * 10;
                    const int ln = hh * 16 + (j >> 2);
                    float acc = rb[slot * 32 + ln];
#pragma unroll
                    for (int wv = 1; wv < 8; ++wv) acc += rb[(wv * 10 + slot) * 32 + ln];
                    gst[(g * kWin + u) * kN + j] = acc;
                }
            }
            __syncthreads();
            // ---- write the window's gradients
            for (int e = tid; e < 6 * nt * (kN / 4); e += kThreads) {
                const int g = e / (nt * (kN / 4));
                const int rem = e % (nt * (kN / 4));
                const int u = rem / (kN / 4), n = (rem % (kN / 4)) * 4;
                *reinterpret_cast<float4 *>(gout[g] + base0 + (size_t)(ws + u) * tstride + n) =
                    *reinterpret_cast<const float4 *>(gst + (g * kWin + u) * kN + n);
            }
        }
    }
    if (p.ds0) store_block(G, p.ds0 + sbase, rg, cg);
}

// ------------------------------------------------------------------- decode

template <typename E>
__device__ __forceinline__ void gload4(const E *src, size_t off, float o[4]);
template <>
__device__ __forceinline__ void gload4<float>(const float *src, size_t off, float o[4]) {
    to4(*reinterpret_cast<const float4 *>(src + off), o);
}
template <>
__device__ __forceinline__ void gload4<__nv_bfloat16>(const __nv_bfloat16 *src, size_t off, float o[4]) {
    const uint2 q = *reinterpret_cast<const uint2 *>(src + off);
    o[0] = bf16_lo(q.x); o[1] = bf16_hi(q.x); o[2] = bf16_lo(q.y); o[3] = bf16_hi(q.y);
}

template <typename E>
__global__ void __launch_bounds__(kThreads) wkv7_decode_kernel(const E *__restrict__ rp, const E *__restrict__ wp,
                                                               const E *__restrict__ kp, const E *__restrict__ vp,
                                                               const E *__restrict__ ap, const E *__restrict__ bp,
                                                               float *__restrict__ state, float *__restrict__ y) {
    const int bh = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cg = lane & 15, rg = warp * 2 + (lane >> 4);
    const size_t vo = (size_t)bh * kN;
    float s[4][4], r[4], w[4], k[4], a[4], b[4], v[4], sa[4], q[4];
    load_block(s, state + vo * kN, rg, cg);
    gload4(wp, vo + cg * 4, w);
    gload4(kp, vo + cg * 4, k);
    gload4(ap, vo + cg * 4, a);
    gload4(bp, vo + cg * 4, b);
    gload4(vp, vo + rg * 4, v);
    gload4(rp, vo + cg * 4, r);
    step(s, w, k, a, b, v, sa, lane);
    store_block(s, state + vo * kN, rg, cg);
    dot_rows(s, r, q);
    const float yv = reduce_rows(q, lane);
    if ((lane & 3) == 0) y[vo + rg * 4 + reduced_row(lane)] = yv;
}

template <typename Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_forward_plain(const SeqArgs &p, cudaStream_t st) {
    const int grid = p.B * p.H;
    if (p.dtype == 1) {
        const size_t sm = 2 * 6 * kChunk * kN * sizeof(__nv_bfloat16) + 2 * kChunk * kN * sizeof(float);
        wkv7_fwd_plain_kernel<__nv_bfloat16><<<grid, kThreads, sm, st>>>(p);
    } else {
        const size_t sm = 2 * 6 * kChunk * kN * sizeof(float) + 2 * kChunk * kN * sizeof(float);
        cudaError_t e = set_smem(wkv7_fwd_plain_kernel<float>, sm);
        if (e != cudaSuccess) return e;
        wkv7_fwd_plain_kernel<float><<<grid, kThreads, sm, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_backward_plain(const SeqArgs &p, cudaStream_t st) {
    const int grid = p.B * p.H;
    cudaError_t e;
    if (p.dtype == 1) {
        const size_t sm = BwdSmem::total<__nv_bfloat16>();
        if ((e = set_smem(wkv7_bwd_plain_kernel<__nv_bfloat16>, sm)) != cudaSuccess) return e;
        wkv7_bwd_plain_kernel<__nv_bfloat16><<<grid, kThreads, sm, st>>>(p);
    } else {
        const size_t sm = BwdSmem::total<float>();
        if ((e = set_smem(wkv7_bwd_plain_kernel<float>, sm)) != cudaSuccess) return e;
        wkv7_bwd_plain_kernel<float><<<grid, kThreads, sm, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_step(int B, int H, int dtype, const void *r, const void *w, const void *k,
                               const void *v, const void *a, const void *b, float *state, float *y,
                               cudaStream_t st) {
    const int grid = B * H;
    if (dtype == 1) {
        using E = __nv_bfloat16;
        wkv7_decode_kernel<E><<<grid, kThreads, 0, st>>>((const E *)r, (const E *)w, (const E *)k, (const E *)v,
                                                         (const E *)a, (const E *)b, state, y);
    } else {
        wkv7_decode_kernel<float><<<grid, kThreads, 0, st>>>((const float *)r, (const float *)w, (const float *)k,
                                                             (const float *)v, (const float *)a, (const float *)b,
                                                             state, y);
    }
    return cudaGetLastError();
}

}  // namespace wkv7
