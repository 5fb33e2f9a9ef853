// The exact per-token backward of one chunk, shared by the chunked backward
// kernels (the chunks whose decays the factorised form cannot divide by),
// and the warp reductions it uses.
#pragma once
#include "wkv7_chunk_common.cuh"

namespace wkv7 {
namespace chunk {

constexpr int NT = 128;  // threads of a chunked-kernel CTA (4 warps)
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(kFull, x, 1);
    x += __shfl_xor_sync(kFull, x, 2);
    return x;
}
// Sum over the 8 lanes that share q (the g index), i.e. over 8 value rows.
__device__ __forceinline__ float rows_sum(float x) {
    x += __shfl_xor_sync(kFull, x, 4);
    x += __shfl_xor_sync(kFull, x, 8);
    x += __shfl_xor_sync(kFull, x, 16);
    return x;
}

// Exact per-token backward of one chunk (decay underflow, or a decay small
// enough that dividing by it would amplify rounding).  G (registers, rows
// rA/rB, columns 8nt+2q+{0,1}) enters as dL/dS_C and leaves as dL/dS_0.  The
// chunk's start state is read from S0s (row stride S0S floats; shared or
// global memory), the chunk's S_{t-1} is kept in Sps ([64][SP] fp32) and the
// column partial sums in red (5 x 4 x 64 fp32).  Writes all six gradients of
// the chunk's tokens and returns, per lane, the dw carry for columns jA/jB of
// the key-row layout (w_0 o dw_0 + a_0 o da_0).
// kGN: the output epilogue's own terms join dv, dr, dk: gpost ([C][SP]) holds
// do s per (token, value), dsv the per-token sum_j do_j v_j, rkh the head's r_k.
template <typename E, bool kP, int S0S, bool kGN = false>
__device__ void bwd_chunk_exact(const E *raw, const float *dys, const float *S0s, float *Sps, float *red,
                                float G[8][4], int nv, const SeqArgs &p, size_t base0, size_t tstride, int t0,
                                float &carryA, float &carryB, const float *gpost = nullptr,
                                const float *dsv = nullptr, const float *rkh = nullptr) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q = lane & 3;
    const int rA = warp * 16 + g, rB = rA + 8;
    for (int t = nv - 1; t >= 0; --t) {
        // replay S_0 -> S_{t-1} (kept in registers), recording nothing
        float S[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float2 x = *reinterpret_cast<const float2 *>(S0s + rA * S0S + 8 * nt + 2 * q);
            const float2 z = *reinterpret_cast<const float2 *>(S0s + rB * S0S + 8 * nt + 2 * q);
            S[nt][0] = x.x; S[nt][1] = x.y; S[nt][2] = z.x; S[nt][3] = z.y;
        }
        float sa0 = 0.f, sa1 = 0.f;
        for (int u = 0; u <= t; ++u) {
            sa0 = 0.f; sa1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j = 8 * nt + 2 * q;
                const float a0 = in_a<kP>(raw, u, j), a1 = in_a<kP>(raw, u, j + 1);
                sa0 = __fmaf_rn(S[nt][0], a0, __fmaf_rn(S[nt][1], a1, sa0));
                sa1 = __fmaf_rn(S[nt][2], a0, __fmaf_rn(S[nt][3], a1, sa1));
            }
            sa0 = quad_sum(sa0);
            sa1 = quad_sum(sa1);
            if (u == t) {  // keep S_{t-1} for dw and da
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    *reinterpret_cast<float2 *>(Sps + rA * SP + 8 * nt + 2 * q) = make_float2(S[nt][0], S[nt][1]);
                    *reinterpret_cast<float2 *>(Sps + rB * SP + 8 * nt + 2 * q) = make_float2(S[nt][2], S[nt][3]);
                }
            }
            const float v0 = ld_raw(raw, VV, u, rA), v1 = ld_raw(raw, VV, u, rB);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = 8 * nt + 2 * q + e;
                    const float wv = in_w<kP>(raw, u, j), kv = ld_raw(raw, VK, u, j), bv = in_b<kP>(raw, u, j);
                    S[nt][e] = __fmaf_rn(S[nt][e], wv, __fmaf_rn(sa0, bv, __fmul_rn(v0, kv)));
                    S[nt][2 + e] = __fmaf_rn(S[nt][2 + e], wv, __fmaf_rn(sa1, bv, __fmul_rn(v1, kv)));
                }
        }
        // now S = S_t, sa0/sa1 = sa_t for rows rA/rB
        const float dy0 = dys[t * SP + rA], dy1 = dys[t * SP + rB];
        const float v0 = ld_raw(raw, VV, t, rA), v1 = ld_raw(raw, VV, t, rB);
        float dv0 = 0.f, dv1 = 0.f, ds0 = 0.f, ds1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * nt + 2 * q + e;
                const float rv = ld_raw(raw, VR, t, j), kv = ld_raw(raw, VK, t, j), bv = in_b<kP>(raw, t, j);
                G[nt][e] = __fmaf_rn(dy0, rv, G[nt][e]);
                G[nt][2 + e] = __fmaf_rn(dy1, rv, G[nt][2 + e]);
                dv0 = __fmaf_rn(G[nt][e], kv, dv0);
                dv1 = __fmaf_rn(G[nt][2 + e], kv, dv1);
                ds0 = __fmaf_rn(G[nt][e], bv, ds0);
                ds1 = __fmaf_rn(G[nt][2 + e], bv, ds1);
            }
        dv0 = quad_sum(dv0); dv1 = quad_sum(dv1);
        ds0 = quad_sum(ds0); ds1 = quad_sum(ds1);
        if (q == 0) {
            p.dv[base0 + (size_t)(t0 + t) * tstride + rA] = dv0 + (kGN ? gpost[t * SP + rA] : 0.f);
            p.dv[base0 + (size_t)(t0 + t) * tstride + rB] = dv1 + (kGN ? gpost[t * SP + rB] : 0.f);
        }
        __syncthreads();  // S_{t-1} visible in Sps
        // column partials over this lane's two rows, reduced over the warp's 16 rows
        // red layout: [grad 0..4][warp][64]; grads: dr, dk, db, dw, da
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * nt + 2 * q + e;
                const float spA = Sps[rA * SP + j], spB = Sps[rB * SP + j];
                float x[5];
                x[0] = __fmaf_rn(S[nt][e], dy0, __fmul_rn(S[nt][2 + e], dy1));
                x[1] = __fmaf_rn(G[nt][e], v0, __fmul_rn(G[nt][2 + e], v1));
                x[2] = __fmaf_rn(G[nt][e], sa0, __fmul_rn(G[nt][2 + e], sa1));
                x[3] = __fmaf_rn(G[nt][e], spA, __fmul_rn(G[nt][2 + e], spB));
                x[4] = __fmaf_rn(spA, ds0, __fmul_rn(spB, ds1));
#pragma unroll
                for (int m = 0; m < 5; ++m) {
                    const float s = rows_sum(x[m]);
                    if (g == 0) red[(m * 4 + warp) * 64 + j] = s;
                }
            }
        // carried gradient to S_{t-1}
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * nt + 2 * q + e;
                const float wv = in_w<kP>(raw, t, j), av = in_a<kP>(raw, t, j);
                G[nt][e] = __fmaf_rn(G[nt][e], wv, __fmul_rn(ds0, av));
                G[nt][2 + e] = __fmaf_rn(G[nt][2 + e], wv, __fmul_rn(ds1, av));
            }
        __syncthreads();
        if constexpr (kP) {  // gradients of the producers' inputs: dw_pre, dkk, davec (k_wdecay_bwd, k_comp_keymod)
            for (int j = tid; j < 64; j += NT) {
                float s5[5];
#pragma unroll
                for (int m = 0; m < 5; ++m)
                    s5[m] = red[(m * 4 + 0) * 64 + j] + red[(m * 4 + 1) * 64 + j] + red[(m * 4 + 2) * 64 + j] +
                            red[(m * 4 + 3) * 64 + j];
                const size_t o = base0 + (size_t)(t0 + t) * tstride + j;
                const float sg = sigmoid_f(ld_raw(raw, VW, t, j)), kkv = ld_raw(raw, VA, t, j), avv = ld_raw(raw, VB, t, j);
                p.dr[o] = s5[0];
                p.dk[o] = s5[1];
                p.db[o] = kkv * s5[2];
                p.dw[o] = s5[3] * in_w<kP>(raw, t, j) * (-kDecayScale) * sg * (1.f - sg);
                p.da[o] = avv * s5[2] - s5[4];
            }
        } else {
            float *outs[5] = {p.dr, p.dk, p.db, p.dw, p.da};
            for (int o = tid; o < 5 * 64; o += NT) {
                const int m = o >> 6, j = o & 63;
                float s = red[(m * 4 + 0) * 64 + j] + red[(m * 4 + 1) * 64 + j] + red[(m * 4 + 2) * 64 + j] +
                          red[(m * 4 + 3) * 64 + j];
                if constexpr (kGN) {  // the bonus's dr = ds k r_k, dk = ds r r_k
                    if (m == 0) s += dsv[t] * ld_raw(raw, VK, t, j) * rkh[j];
                    if (m == 1) s += dsv[t] * ld_raw(raw, VR, t, j) * rkh[j];
                }
                outs[m][base0 + (size_t)(t0 + t) * tstride + j] = s;
            }
        }
        if (t == 0) {  // dw carry into the previous chunk: w_0 o dw_0 + a_0 o da_0
            const int jA = warp * 16 + g, jB = jA + 8;
            float cA = 0.f, cB = 0.f;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
                cA += in_w<kP>(raw, 0, jA) * red[(3 * 4 + w4) * 64 + jA] + in_a<kP>(raw, 0, jA) * red[(4 * 4 + w4) * 64 + jA];
                cB += in_w<kP>(raw, 0, jB) * red[(3 * 4 + w4) * 64 + jB] + in_a<kP>(raw, 0, jB) * red[(4 * 4 + w4) * 64 + jB];
            }
            carryA = cA;
            carryB = cB;
        }
        __syncthreads();
    }
}

// The same chunk for the state gradient alone: G enters as dL/dS_C and
// leaves as dL/dS_0 through the operations of bwd_chunk_exact, in its order
// (G += dy_t r_t^T, dsa = G b_t, G <- G diag(w_t) + dsa a_t^T), so the result
// is bit-identical to it.  dS does not depend on the state: no start state,
// no k or v, no per-token gradient and no block barrier.
template <typename E, bool kP>
__device__ void bwd_chunk_exact_state(const E *raw, const float *dys, float G[8][4], int nv) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q = lane & 3;
    const int rA = warp * 16 + g, rB = rA + 8;
    for (int t = nv - 1; t >= 0; --t) {
        const float dy0 = dys[t * SP + rA], dy1 = dys[t * SP + rB];
        float ds0 = 0.f, ds1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * nt + 2 * q + e;
                const float rv = ld_raw(raw, VR, t, j), bv = in_b<kP>(raw, t, j);
                G[nt][e] = __fmaf_rn(dy0, rv, G[nt][e]);
                G[nt][2 + e] = __fmaf_rn(dy1, rv, G[nt][2 + e]);
                ds0 = __fmaf_rn(G[nt][e], bv, ds0);
                ds1 = __fmaf_rn(G[nt][2 + e], bv, ds1);
            }
        ds0 = quad_sum(ds0);
        ds1 = quad_sum(ds1);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * nt + 2 * q + e;
                const float wv = in_w<kP>(raw, t, j), av = in_a<kP>(raw, t, j);
                G[nt][e] = __fmaf_rn(G[nt][e], wv, __fmul_rn(ds0, av));
                G[nt][2 + e] = __fmaf_rn(G[nt][2 + e], wv, __fmul_rn(ds1, av));
            }
    }
}

}  // namespace chunk
}  // namespace wkv7
