// Chunked WKV7 forward on warp-level tensor cores.
//
// Per (b,h) the recurrence S_t = S_{t-1} diag(w_t) + (S_{t-1} a_t) b_t^T
// + v_t k_t^T, y_t = S_t r_t (layouts of the "Foundry/cuda_kernels/timemix.cu"
// page) is evaluated 16 tokens at a time.  Inside a chunk, with the
// cumulative decay d_t = w_1 o ... o w_t (per key column) and the chunk-start
// state S_0, unrolling the recurrence gives
//     S_t = (S_0 + sum_{s<=t} sa_s (b_s/d_s)^T + v_s (k_s/d_s)^T) diag(d_t),
// so the chunk's sa_t = S_{t-1} a_t solve a unit triangular 16x16 system and
// every state-dependent quantity is a dense contraction:
//     SA  = S_0 A' + V M_k'              (A' = A^ W,  M_k' = M_k W)
//     Y   = S_0 R' + V Q'                (R' = R^ + A' Q_b,  Q' = Q_k + M_k' Q_b)
//     S_C = S_0 diag(d_C) + SA Bbar^T + V Kbar^T
// with A^ = [a_t o d_{t-1}], R^ = [r_t o d_t], B~ = [b_s / d_s], K~ = [k_s / d_s],
// Bbar = B~ diag(d_C), Kbar = K~ diag(d_C), the Gram blocks
// M_b[s][t] = b~_s.a^_t (s<t), M_k[s][t] = k~_s.a^_t (s<t), Q_b[s][t] = b~_s.r^_t
// (s<=t), Q_k[s][t] = k~_s.r^_t (s<=t), and W = (I - M_b)^{-1}.  The matrices
// that do not involve S_0 are built per chunk in shared memory; the state
// products run on mma.sync bf16 with split (hi+lo) operands and fp32
// accumulation.  The state lives in registers as MMA accumulators: warp w owns
// rows 16w..16w+15.
//
// A chunk whose cumulative decay underflows (min d_C < 1e-20, e.g. w = 0)
// cannot use 1/d_s; it takes the exact per-token recurrence instead, on the
// same register layout.
#include "wkv7_internal.cuh"
#include "wkv7_mma.cuh"

namespace wkv7 {
namespace {

constexpr int C = 16;              // tokens per chunk
constexpr int NT = 128;            // 4 warps
constexpr int SP = 72;             // row stride (floats) of [token][key] arrays
constexpr int GS = 33;             // row stride of the 32x32 Gram
constexpr int QS = 36;             // row stride of the [s][32] V-side operand
constexpr int WS = 17;             // row stride of W
constexpr int GU = (32 * GS > C * SP) ? 32 * GS : C * SP;  // Gram / y staging union
constexpr float kTiny = 1e-20f;
enum { VR = 0, VW = 1, VK = 2, VV = 3, VA = 4, VB = 5 };

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

template <typename E>
__device__ __forceinline__ float ld_raw(const E *raw, int vec, int t, int j);
template <>
__device__ __forceinline__ float ld_raw<float>(const float *raw, int vec, int t, int j) {
    return raw[(vec * C + t) * 64 + j];
}
template <>
__device__ __forceinline__ float ld_raw<__nv_bfloat16>(const __nv_bfloat16 *raw, int vec, int t, int j) {
    return __bfloat162float(raw[(vec * C + t) * 64 + j]);
}

// cp.async copies of the six input vectors of tokens [t0, t0 + C) into raw
// [vec][C][64]; tokens at or beyond `nvalid` are zero-filled.
template <typename E>
__device__ __forceinline__ void stage_chunk(E *raw, const E *const (&src)[6], size_t base, size_t tstride,
                                            int nvalid) {
    constexpr int P = 16 / sizeof(E);
    constexpr int per_tok = 64 / P;
    constexpr int per_vec = C * per_tok;
#pragma unroll
    for (int vv = 0; vv < 6; ++vv) {
        for (int e = threadIdx.x; e < per_vec; e += NT) {
            const int u = e / per_tok, n = (e % per_tok) * P;
            const bool ok = u < nvalid;
            const E *g = ok ? src[vv] + base + (size_t)u * tstride + n : src[vv];
            cp_async16(raw + (vv * C + u) * 64 + n, g, ok ? 16 : 0);
        }
    }
}

__device__ __forceinline__ float2 f2(const float *a, int row, int col) {
    return *reinterpret_cast<const float2 *>(a + row * SP + col);
}

template <typename E>
__host__ __device__ constexpr size_t raw_bytes() { return (size_t)6 * C * 64 * sizeof(E); }
constexpr size_t kFloatsAfterRaw = 5 * C * SP + GU + C * WS + C * QS;

template <typename E>
__global__ void __launch_bounds__(NT) wkv7_fwd_chunk_kernel(SeqArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);
    float *ah = reinterpret_cast<float *>(smem + raw_bytes<E>());  // a o d_{t-1}, then A'
    float *rh = ah + C * SP;                                          // r o d_t, then R'
    float *bt = rh + C * SP;                                          // b / d_t
    float *kt = bt + C * SP;                                          // k / d_t
    float *dd = kt + C * SP;                                          // d_t
    float *G = dd + C * SP;                                           // Gram [32][GS]; later y staging
    float *ys = G;
    float *Wm = G + GU;                                               // W [16][WS]
    float *QM = Wm + C * WS;                                          // [s][0..15] = Q', [s][16..31] = M_k'

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int bh = blockIdx.x, bi = bh / p.H, h = bh % p.H;
    const size_t tstride = (size_t)p.H * 64;
    const size_t base0 = ((size_t)bi * p.T * p.H + h) * 64;
    const size_t sbase = (size_t)bh * 64 * 64;
    const int row0 = warp * 16;
    const int rA = row0 + g, rB = row0 + g + 8;  // the two state rows this lane holds

    float S[8][4];  // S[rA][8nt+2q..+1] = S[nt][0..1], S[rB][..] = S[nt][2..3]
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        if (p.s0) {
            const float2 x = *reinterpret_cast<const float2 *>(p.s0 + sbase + rA * 64 + 8 * nt + 2 * q);
            const float2 z = *reinterpret_cast<const float2 *>(p.s0 + sbase + rB * 64 + 8 * nt + 2 * q);
            S[nt][0] = x.x; S[nt][1] = x.y; S[nt][2] = z.x; S[nt][3] = z.y;
        } else {
            S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
        }
    }

    const E *const src[6] = {static_cast<const E *>(p.r), static_cast<const E *>(p.w), static_cast<const E *>(p.k),
                             static_cast<const E *>(p.v), static_cast<const E *>(p.a), static_cast<const E *>(p.b)};
    const int nchunks = (p.T + C - 1) / C;
    stage_chunk<E>(raw, src, base0, tstride, min(C, p.T));
    cp_async_commit();

    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        cp_async_wait_all();
        __syncthreads();

        if (p.ckpt && t0 % p.L == 0) {
            float *dst = p.ckpt + ((size_t)bh * p.nck + t0 / p.L) * 64 * 64;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                *reinterpret_cast<float2 *>(dst + rA * 64 + 8 * nt + 2 * q) = make_float2(S[nt][0], S[nt][1]);
                *reinterpret_cast<float2 *>(dst + rB * 64 + 8 * nt + 2 * q) = make_float2(S[nt][2], S[nt][3]);
            }
        }

        // cumulative decay per key column (padding tokens decay by 1)
        bool tiny = false;
        if (tid < 64) {
            float dc = 1.f;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                const float wv = t < nv ? ld_raw(raw, VW, t, tid) : 1.f;
                dc = __fmul_rn(dc, wv);
                dd[t * SP + tid] = dc;
            }
            tiny = !(dc >= kTiny);
        }
        const bool exact = __syncthreads_or(tiny);

        if (!exact) {
            // decay-scaled chunk vectors
            for (int e = tid; e < C * 64; e += NT) {
                const int t = e >> 6, j = e & 63;
                const float d = dd[t * SP + j];
                const float dp = t ? dd[(t - 1) * SP + j] : 1.f;
                const float inv = __frcp_rn(d);
                ah[t * SP + j] = ld_raw(raw, VA, t, j) * dp;
                rh[t * SP + j] = ld_raw(raw, VR, t, j) * d;
                bt[t * SP + j] = ld_raw(raw, VB, t, j) * inv;
                kt[t * SP + j] = ld_raw(raw, VK, t, j) * inv;
            }
            // this warp's V block as an A operand: rows = state rows, k = token
            const AFrag va = make_a(make_float2(ld_raw(raw, VV, 2 * q, rA), ld_raw(raw, VV, 2 * q + 1, rA)),
                                    make_float2(ld_raw(raw, VV, 2 * q, rB), ld_raw(raw, VV, 2 * q + 1, rB)),
                                    make_float2(ld_raw(raw, VV, 2 * q + 8, rA), ld_raw(raw, VV, 2 * q + 9, rA)),
                                    make_float2(ld_raw(raw, VV, 2 * q + 8, rB), ld_raw(raw, VV, 2 * q + 9, rB)));
            __syncthreads();
            if (c + 1 < nchunks) stage_chunk<E>(raw, src, base0 + (size_t)(t0 + C) * tstride, tstride, min(C, p.T - t0 - C));
            cp_async_commit();

            // Gram [B~;K~] [A^;R^]^T over the 64 key columns: warp -> (m-tile, two n-tiles)
            {
                const int mt = warp >> 1;
                const float *As = mt ? kt : bt;
                float acc[2][4] = {};
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const AFrag af = make_a(f2(As, g, 16 * kk + 2 * q), f2(As, g + 8, 16 * kk + 2 * q),
                                            f2(As, g, 16 * kk + 2 * q + 8), f2(As, g + 8, 16 * kk + 2 * q + 8));
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int nt = 2 * (warp & 1) + u;
                        const float *Bs = nt < 2 ? ah : rh;
                        const int tt = 8 * (nt & 1) + g;
                        mma3(acc[u], af, make_b(f2(Bs, tt, 16 * kk + 2 * q), f2(Bs, tt, 16 * kk + 2 * q + 8)));
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int col = 8 * (2 * (warp & 1) + u) + 2 * q, row = 16 * mt + g;
                    G[row * GS + col] = acc[u][0];
                    G[row * GS + col + 1] = acc[u][1];
                    G[(row + 8) * GS + col] = acc[u][2];
                    G[(row + 8) * GS + col + 1] = acc[u][3];
                }
            }
            __syncthreads();

            // W = (I - M_b)^{-1}, lane t builds column t by back substitution
            if (warp == 0 && lane < C) {
                const int t = lane;
                float wc[C];
#pragma unroll
                for (int s = C - 1; s >= 0; --s) {
                    float acc = (s == t) ? 1.f : 0.f;
#pragma unroll
                    for (int u = s + 1; u < C; ++u) acc = __fmaf_rn(G[s * GS + u], wc[u], acc);
                    wc[s] = acc;
                }
#pragma unroll
                for (int s = 0; s < C; ++s) Wm[s * WS + t] = wc[s];
            }
            __syncthreads();

            if (tid < 64) {  // A' = A^ W, in place, one key column per thread
                const int j = tid;
                float col[C];
#pragma unroll
                for (int s = 0; s < C; ++s) col[s] = ah[s * SP + j];
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    float acc = 0.f;
#pragma unroll
                    for (int s = 0; s <= t; ++s) acc = __fmaf_rn(col[s], Wm[s * WS + t], acc);
                    ah[t * SP + j] = acc;
                }
            } else {  // M_k' = M_k W (strictly upper) into QM[s][16 + t]
                for (int o = tid - 64; o < C * C; o += 64) {
                    const int s = o >> 4, t = o & 15;
                    float acc = 0.f;
                    for (int u = s + 1; u <= t; ++u) acc = __fmaf_rn(G[(16 + s) * GS + u], Wm[u * WS + t], acc);
                    QM[s * QS + 16 + t] = acc;
                }
            }
            __syncthreads();
            // R' = R^ + A' Q_b (in place) and Q' = Q_k + M_k' Q_b
            for (int e = tid; e < C * 64; e += NT) {
                const int t = e >> 6, j = e & 63;
                float acc = rh[t * SP + j];
                for (int s = 0; s <= t; ++s) acc = __fmaf_rn(ah[s * SP + j], G[s * GS + 16 + t], acc);
                rh[t * SP + j] = acc;
            }
            for (int o = tid; o < C * C; o += NT) {
                const int s = o >> 4, t = o & 15;
                float acc = s <= t ? G[(16 + s) * GS + 16 + t] : 0.f;
                for (int u = s + 1; u <= t; ++u) acc = __fmaf_rn(QM[s * QS + 16 + u], G[u * GS + 16 + t], acc);
                QM[s * QS + t] = acc;
            }
            __syncthreads();

            // [Y | SA] = S_0 [R' | A'] + V [Q' | M_k']
            float ya[4][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const AFrag sf = a_from_acc(S, kk);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const float *X = nt < 2 ? rh : ah;
                    const int tt = 8 * (nt & 1) + g;
                    mma3(ya[nt], sf, make_b(f2(X, tt, 16 * kk + 2 * q), f2(X, tt, 16 * kk + 2 * q + 8)));
                }
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n = 8 * nt + g;
                mma3(ya[nt], va,
                     make_b(make_float2(QM[(2 * q) * QS + n], QM[(2 * q + 1) * QS + n]),
                            make_float2(QM[(2 * q + 8) * QS + n], QM[(2 * q + 9) * QS + n])));
            }

            // S_C = S_0 diag(d_C) + [SA | V] [Bbar^T ; Kbar^T]
            const AFrag saf = make_a(make_float2(ya[2][0], ya[2][1]), make_float2(ya[2][2], ya[2][3]),
                                     make_float2(ya[3][0], ya[3][1]), make_float2(ya[3][2], ya[3][3]));
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j0 = 8 * nt + 2 * q;
                const float dc0 = dd[(C - 1) * SP + j0], dc1 = dd[(C - 1) * SP + j0 + 1];
                S[nt][0] *= dc0; S[nt][1] *= dc1; S[nt][2] *= dc0; S[nt][3] *= dc1;
                const int jn = 8 * nt + g;
                const float dcn = dd[(C - 1) * SP + jn];
                const BFrag bb = make_b(make_float2(bt[(2 * q) * SP + jn] * dcn, bt[(2 * q + 1) * SP + jn] * dcn),
                                        make_float2(bt[(2 * q + 8) * SP + jn] * dcn, bt[(2 * q + 9) * SP + jn] * dcn));
                const BFrag kb = make_b(make_float2(kt[(2 * q) * SP + jn] * dcn, kt[(2 * q + 1) * SP + jn] * dcn),
                                        make_float2(kt[(2 * q + 8) * SP + jn] * dcn, kt[(2 * q + 9) * SP + jn] * dcn));
                mma3(S[nt], saf, bb);
                mma3(S[nt], va, kb);
            }
            // y of the chunk -> staging [t][row]
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t = 8 * nt + 2 * q;
                ys[t * SP + rA] = ya[nt][0];
                ys[(t + 1) * SP + rA] = ya[nt][1];
                ys[t * SP + rB] = ya[nt][2];
                ys[(t + 1) * SP + rB] = ya[nt][3];
            }
        } else {
            // exact per-token recurrence for a chunk whose decay underflows
            for (int t = 0; t < nv; ++t) {
                float sa0 = 0.f, sa1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int j = 8 * nt + 2 * q;
                    const float a0 = ld_raw(raw, VA, t, j), a1 = ld_raw(raw, VA, t, j + 1);
                    sa0 = __fmaf_rn(S[nt][0], a0, __fmaf_rn(S[nt][1], a1, sa0));
                    sa1 = __fmaf_rn(S[nt][2], a0, __fmaf_rn(S[nt][3], a1, sa1));
                }
                sa0 += __shfl_xor_sync(0xffffffffu, sa0, 1);
                sa0 += __shfl_xor_sync(0xffffffffu, sa0, 2);
                sa1 += __shfl_xor_sync(0xffffffffu, sa1, 1);
                sa1 += __shfl_xor_sync(0xffffffffu, sa1, 2);
                const float v0 = ld_raw(raw, VV, t, rA), v1 = ld_raw(raw, VV, t, rB);
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 8 * nt + 2 * q + e;
                        const float wv = ld_raw(raw, VW, t, j), kv = ld_raw(raw, VK, t, j);
                        const float bv = ld_raw(raw, VB, t, j), rv = ld_raw(raw, VR, t, j);
                        S[nt][e] = __fmaf_rn(S[nt][e], wv, __fmaf_rn(sa0, bv, __fmul_rn(v0, kv)));
                        S[nt][2 + e] = __fmaf_rn(S[nt][2 + e], wv, __fmaf_rn(sa1, bv, __fmul_rn(v1, kv)));
                        y0 = __fmaf_rn(S[nt][e], rv, y0);
                        y1 = __fmaf_rn(S[nt][2 + e], rv, y1);
                    }
                }
                y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
                y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
                y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
                y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
                if (q == 0) {
                    ys[t * SP + rA] = y0;
                    ys[t * SP + rB] = y1;
                }
            }
            __syncthreads();
            if (c + 1 < nchunks) stage_chunk<E>(raw, src, base0 + (size_t)(t0 + C) * tstride, tstride, min(C, p.T - t0 - C));
            cp_async_commit();
        }
        __syncthreads();
        for (int e = tid; e < nv * 16; e += NT) {
            const int t = e >> 4, n = (e & 15) * 4;
            *reinterpret_cast<float4 *>(p.y + base0 + (size_t)(t0 + t) * tstride + n) =
                *reinterpret_cast<const float4 *>(ys + t * SP + n);
        }
    }
    cp_async_wait_all();
    if (p.sT) {
        float *dst = p.sT + sbase;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<float2 *>(dst + rA * 64 + 8 * nt + 2 * q) = make_float2(S[nt][0], S[nt][1]);
            *reinterpret_cast<float2 *>(dst + rB * 64 + 8 * nt + 2 * q) = make_float2(S[nt][2], S[nt][3]);
        }
    }
}

}  // namespace

bool forward_chunk_supported(const SeqArgs &p) { return p.L % C == 0; }

cudaError_t launch_forward_chunk(const SeqArgs &p, cudaStream_t st) {
    const int grid = p.B * p.H;
    cudaError_t e;
    if (p.dtype == 1) {
        const size_t sm = raw_bytes<__nv_bfloat16>() + kFloatsAfterRaw * sizeof(float);
        if ((e = cudaFuncSetAttribute(wkv7_fwd_chunk_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sm)) != cudaSuccess)
            return e;
        wkv7_fwd_chunk_kernel<__nv_bfloat16><<<grid, NT, sm, st>>>(p);
    } else {
        const size_t sm = raw_bytes<float>() + kFloatsAfterRaw * sizeof(float);
        if ((e = cudaFuncSetAttribute(wkv7_fwd_chunk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sm)) != cudaSuccess)
            return e;
        wkv7_fwd_chunk_kernel<float><<<grid, NT, sm, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace wkv7
