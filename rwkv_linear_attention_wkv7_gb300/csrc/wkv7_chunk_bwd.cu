// Chunked WKV7 backward on warp-level tensor cores.
//
// The adjoint of the recurrence (the "WKV kernel backward" block of
// accumulate_token_step_gradients on the "infotheory/backends/rwkvzip/rwkv7/
// model.rs" page: dS carried backwards, scaled by w per key column plus a
// rank-1 term along a) is evaluated one 16-token chunk at a time, last chunk
// first, from the chunk-start states the forward checkpointed (stride 16, the
// replay-from-checkpoint scheme of online_train_segment_tbptt on that page).
//
// With the chunk notation of wkv7_chunk_common.cuh, G = dL/dS_C the gradient
// arriving from later tokens, and Gd = G diag(d_C), the gradient of the state
// after token t is  H_t = [Gd + sum_{s>=t} dy_s r^_s^T + sum_{s>t} dsa_s a^_s^T] diag(1/d_t),
// which makes every gradient a dense contraction:
//   SA          = S_0 A' + V M_k'                          (recomputed)
//   [DV | DSA]  = G [K' | B'] + DY [Q'^T | Q_b'^T]           K' = Kbar + Bbar M_k'^T,
//                                                             B' = Bbar W^T, Q_b' = W Q_b
//   Gam         = [SA | V]^T [DY | DSA]                      (32 x 32)
//   [DR | DA]   = [d | d_prev] o (S_0^T [DY | DSA] + [B~ | K~] mask(Gam))
//   [DK | DB]   = (1/d) o (Gd^T [V | SA] + [R^ | A^] mask(Gam^T))
//   G_prev      = Gd + [DY | DSA] [R^ | A^]^T
// dw needs no contraction of its own: summing H_t o S_t over the value rows
// in two ways gives, per key column,
//   w_t o dw_t = r_t o dr_t - b_t o db_t - k_t o dk_t + (w o dw + a o da)_{t+1},
// a reverse running sum whose value past the last token is diag(dsT^T sT).
// Chunks whose decay underflows take an exact per-token path that replays
// the chunk from its checkpoint.
#include "wkv7_chunk_common.cuh"

namespace wkv7 {
namespace {
using namespace chunk;

constexpr int NT = 128;
constexpr int QS = 36;   // QM [C][QS]: M_k' in columns 16..31
constexpr int QQS = 24;  // QQ [32][QQS]: rows 0..15 = Q', rows 16..31 = W Q_b
constexpr unsigned kFull = 0xffffffffu;

// Float offsets of the shared-memory carve-up (after the raw input block).
constexpr int O_DY = 0;                 // dy       [C][SP]
constexpr int O_S0 = O_DY + C * SP;     // S_0      [64][SP]
constexpr int O_GD = O_S0 + 64 * SP;    // G d_C    [64][SP]  (exact path: S_{t-1})
constexpr int O_AH = O_GD + 64 * SP;    // a^       [C][SP]
constexpr int O_RH = O_AH + C * SP;     // r^
constexpr int O_BT = O_RH + C * SP;     // b~
constexpr int O_KT = O_BT + C * SP;     // k~
constexpr int O_DD = O_KT + C * SP;     // d
constexpr int O_VT = O_DD + C * SP;     // v (fp32)
constexpr int O_KB = O_VT + C * SP;     // [K'; B'] [32][SP]
constexpr int O_GM = O_KB + 32 * SP;    // Gram, then Gam [32][GS]
constexpr int O_WM = O_GM + 32 * GS;    // W [C][WS]
constexpr int O_QM = O_WM + C * WS;     // M_k' [C][QS]
constexpr int O_QQ = O_QM + C * QS;     // [32][QQS]
constexpr int O_SA = O_QQ + 32 * QQS;   // SA (token-major [t][i]) [C][SP]
constexpr int O_DS = O_SA + C * SP;     // A' until SA is known, then DSA (token-major) [C][SP]
constexpr int kFloats = O_DS + C * SP;
// Reduction scratch aliases buffers idle at the time: the exact path uses the
// [K'; B'] block ([5][4][64] floats), the dsT o sT start uses the DSA block.
static_assert(5 * 4 * 64 <= 32 * SP, "exact-path scratch must fit the [K'; B'] block");
static_assert(4 * 64 <= C * SP, "dw start scratch must fit the DSA block");

template <typename E>
__host__ __device__ constexpr size_t bwd_smem_bytes() { return raw_bytes<E>() + (size_t)kFloats * sizeof(float); }

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

// Exact per-token backward of one chunk (decay underflow).  G (registers,
// rows rA/rB, columns 8nt+2q+{0,1}) enters as dL/dS_C and leaves as dL/dS_0.
// Writes all six gradients of the chunk's tokens and returns, per lane, the
// dw carry for columns jA/jB of the G3/G4 layout (w_0 o dw_0 + a_0 o da_0).
template <typename E>
__device__ void bwd_chunk_exact(const E *raw, const float *dys, const float *S0s, float *Sps, float *red,
                                float G[8][4], int nv, const SeqArgs &p, size_t base0, size_t tstride, int t0,
                                float &carryA, float &carryB) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q = lane & 3;
    const int rA = warp * 16 + g, rB = rA + 8;
    for (int t = nv - 1; t >= 0; --t) {
        // replay S_0 -> S_{t-1} (kept in registers), recording nothing
        float S[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float2 x = *reinterpret_cast<const float2 *>(S0s + rA * SP + 8 * nt + 2 * q);
            const float2 z = *reinterpret_cast<const float2 *>(S0s + rB * SP + 8 * nt + 2 * q);
            S[nt][0] = x.x; S[nt][1] = x.y; S[nt][2] = z.x; S[nt][3] = z.y;
        }
        float sa0 = 0.f, sa1 = 0.f;
        for (int u = 0; u <= t; ++u) {
            sa0 = 0.f; sa1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j = 8 * nt + 2 * q;
                const float a0 = ld_raw(raw, VA, u, j), a1 = ld_raw(raw, VA, u, j + 1);
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
                    const float wv = ld_raw(raw, VW, u, j), kv = ld_raw(raw, VK, u, j), bv = ld_raw(raw, VB, u, j);
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
                const float rv = ld_raw(raw, VR, t, j), kv = ld_raw(raw, VK, t, j), bv = ld_raw(raw, VB, t, j);
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
            p.dv[base0 + (size_t)(t0 + t) * tstride + rA] = dv0;
            p.dv[base0 + (size_t)(t0 + t) * tstride + rB] = dv1;
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
                const float wv = ld_raw(raw, VW, t, j), av = ld_raw(raw, VA, t, j);
                G[nt][e] = __fmaf_rn(G[nt][e], wv, __fmul_rn(ds0, av));
                G[nt][2 + e] = __fmaf_rn(G[nt][2 + e], wv, __fmul_rn(ds1, av));
            }
        __syncthreads();
        float *outs[5] = {p.dr, p.dk, p.db, p.dw, p.da};
        for (int o = tid; o < 5 * 64; o += NT) {
            const int m = o >> 6, j = o & 63;
            const float s = red[(m * 4 + 0) * 64 + j] + red[(m * 4 + 1) * 64 + j] + red[(m * 4 + 2) * 64 + j] +
                            red[(m * 4 + 3) * 64 + j];
            outs[m][base0 + (size_t)(t0 + t) * tstride + j] = s;
        }
        if (t == 0) {  // dw carry into the previous chunk: w_0 o dw_0 + a_0 o da_0
            const int jA = warp * 16 + g, jB = jA + 8;
            float cA = 0.f, cB = 0.f;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
                cA += ld_raw(raw, VW, 0, jA) * red[(3 * 4 + w4) * 64 + jA] + ld_raw(raw, VA, 0, jA) * red[(4 * 4 + w4) * 64 + jA];
                cB += ld_raw(raw, VW, 0, jB) * red[(3 * 4 + w4) * 64 + jB] + ld_raw(raw, VA, 0, jB) * red[(4 * 4 + w4) * 64 + jB];
            }
            carryA = cA;
            carryB = cB;
        }
        __syncthreads();
    }
}

template <typename E>
__global__ void __launch_bounds__(NT) wkv7_bwd_chunk_kernel(SeqArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);
    float *F = reinterpret_cast<float *>(smem + raw_bytes<E>());
    float *dys = F + O_DY, *S0s = F + O_S0, *Gds = F + O_GD;
    float *ah = F + O_AH, *rh = F + O_RH, *bt = F + O_BT, *kt = F + O_KT, *dd = F + O_DD;
    float *ap = F + O_DS, *vt = F + O_VT, *KB = F + O_KB, *Gm = F + O_GM, *Wm = F + O_WM;
    float *QM = F + O_QM, *QQ = F + O_QQ, *SAt = F + O_SA, *DSt = F + O_DS;
    float *red_exact = KB, *red_start = DSt;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int bh = blockIdx.x, bi = bh / p.H, h = bh % p.H;
    const size_t tstride = (size_t)p.H * 64;
    const size_t base0 = ((size_t)bi * p.T * p.H + h) * 64;
    const size_t sbase = (size_t)bh * 64 * 64;
    const int rA = warp * 16 + g, rB = rA + 8;  // value rows (row-owned products) / key rows (G3, G4)

    float Gh[8][4];  // dL/dS at the current chunk end, rows rA/rB, columns 8nt+2q+{0,1}
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        if (p.dsT) {
            const float2 x = *reinterpret_cast<const float2 *>(p.dsT + sbase + rA * 64 + 8 * nt + 2 * q);
            const float2 z = *reinterpret_cast<const float2 *>(p.dsT + sbase + rB * 64 + 8 * nt + 2 * q);
            Gh[nt][0] = x.x; Gh[nt][1] = x.y; Gh[nt][2] = z.x; Gh[nt][3] = z.y;
        } else {
            Gh[nt][0] = Gh[nt][1] = Gh[nt][2] = Gh[nt][3] = 0.f;
        }
    }
    float carryA = 0.f, carryB = 0.f;  // dw running sum for key columns rA / rB

    const E *const src[6] = {static_cast<const E *>(p.r), static_cast<const E *>(p.w), static_cast<const E *>(p.k),
                             static_cast<const E *>(p.v), static_cast<const E *>(p.a), static_cast<const E *>(p.b)};
    const int nchunks = (p.T + C - 1) / C;
    auto stage_all = [&](int c) {
        const int t0 = c * C, nv = min(C, p.T - t0);
        stage<E, 6, NT>(raw, src, base0 + (size_t)t0 * tstride, tstride, nv);
        stage_rows<NT>(dys, p.dy + base0 + (size_t)t0 * tstride, tstride, C, nv);
        stage_rows<NT>(S0s, p.ckpt_in + ((size_t)bh * p.nck + c) * 64 * 64, 64, 64, 64);
    };
    stage_all(nchunks - 1);
    cp_async_commit();

    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        const bool last = c == nchunks - 1;
        cp_async_wait_all();
        __syncthreads();

        const bool exact = __syncthreads_or(prep_decay(raw, dd, nv));
        if (exact) {
            bwd_chunk_exact<E>(raw, dys, S0s, Gds, red_exact, Gh, nv, p, base0, tstride, t0, carryA, carryB);
            __syncthreads();
            if (c > 0) stage_all(c - 1);
            cp_async_commit();
            continue;
        }

        // ---------------- per-chunk operands (no state involved)
        prep_scaled<E, NT>(raw, dd, ah, rh, bt, kt);
        for (int e = tid; e < C * 64; e += NT) vt[(e >> 6) * SP + (e & 63)] = ld_raw(raw, VV, e >> 6, e & 63);
        __syncthreads();
        prep_gram(ah, rh, bt, kt, Gm);
        __syncthreads();
        prep_inverse(Gm, Wm);
        __syncthreads();
        if (tid < 64) {  // A' = A^ W (separate array: A^ is still needed)
            const int j = tid;
            float col[C];
#pragma unroll
            for (int s = 0; s < C; ++s) col[s] = ah[s * SP + j];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int s = 0; s <= t; ++s) acc = __fmaf_rn(col[s], Wm[s * WS + t], acc);
                ap[t * SP + j] = acc;
            }
        } else {  // M_k' = M_k W
            for (int o = tid - 64; o < C * C; o += 64) {
                const int s = o >> 4, t = o & 15;
                float acc = 0.f;
                for (int u = s + 1; u <= t; ++u) acc = __fmaf_rn(Gm[(16 + s) * GS + u], Wm[u * WS + t], acc);
                QM[s * QS + 16 + t] = acc;
            }
        }
        __syncthreads();
        // Q' (rows 0..15 of QQ) and W Q_b (rows 16..31), both indexed [t][s], nonzero for t <= s
        for (int o = tid; o < 2 * C * C; o += NT) {
            const int which = o >> 8, t = (o >> 4) & 15, s = o & 15;
            float acc = 0.f;
            if (which == 0) {
                if (t <= s) {
                    acc = Gm[(16 + t) * GS + 16 + s];
                    for (int u = t + 1; u <= s; ++u) acc = __fmaf_rn(QM[t * QS + 16 + u], Gm[u * GS + 16 + s], acc);
                }
            } else {
                for (int u = t; u <= s; ++u) acc = __fmaf_rn(Wm[t * WS + u], Gm[u * GS + 16 + s], acc);
            }
            QQ[(16 * which + t) * QQS + s] = acc;
        }
        // K' and B' (token-major, scaled by d_C)
        for (int e = tid; e < C * 64; e += NT) {
            const int t = e >> 6, j = e & 63;
            const float dC = dd[(C - 1) * SP + j];
            float kp = kt[t * SP + j], bp = 0.f;
            for (int s = t + 1; s < C; ++s) kp = __fmaf_rn(bt[s * SP + j], QM[t * QS + 16 + s], kp);
            for (int s = t; s < C; ++s) bp = __fmaf_rn(bt[s * SP + j], Wm[t * WS + s], bp);
            KB[t * SP + j] = kp * dC;
            KB[(16 + t) * SP + j] = bp * dC;
        }
        // G diag(d_C): registers (accumulator init of G_prev) and shared memory (for Gd^T)
        float Gd[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int j0 = 8 * nt + 2 * q;
            const float d0 = dd[(C - 1) * SP + j0], d1 = dd[(C - 1) * SP + j0 + 1];
            Gd[nt][0] = Gh[nt][0] * d0; Gd[nt][1] = Gh[nt][1] * d1;
            Gd[nt][2] = Gh[nt][2] * d0; Gd[nt][3] = Gh[nt][3] * d1;
            *reinterpret_cast<float2 *>(Gds + rA * SP + j0) = make_float2(Gd[nt][0], Gd[nt][1]);
            *reinterpret_cast<float2 *>(Gds + rB * SP + j0) = make_float2(Gd[nt][2], Gd[nt][3]);
        }
        __syncthreads();
        if (c > 0) stage<E, 6, NT>(raw, src, base0 + (size_t)(t0 - C) * tstride, tstride, C);
        cp_async_commit();

        // ---------------- G1: SA = S_0 A' + V M_k'  (rows = value index)
        const AFrag vA = make_a(make_float2(vt[(2 * q) * SP + rA], vt[(2 * q + 1) * SP + rA]),
                                make_float2(vt[(2 * q) * SP + rB], vt[(2 * q + 1) * SP + rB]),
                                make_float2(vt[(2 * q + 8) * SP + rA], vt[(2 * q + 9) * SP + rA]),
                                make_float2(vt[(2 * q + 8) * SP + rB], vt[(2 * q + 9) * SP + rB]));
        const AFrag dyA = make_a(make_float2(dys[(2 * q) * SP + rA], dys[(2 * q + 1) * SP + rA]),
                                 make_float2(dys[(2 * q) * SP + rB], dys[(2 * q + 1) * SP + rB]),
                                 make_float2(dys[(2 * q + 8) * SP + rA], dys[(2 * q + 9) * SP + rA]),
                                 make_float2(dys[(2 * q + 8) * SP + rB], dys[(2 * q + 9) * SP + rB]));
        float sa[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag sf = make_a(f2(S0s, rA, 16 * kk + 2 * q), f2(S0s, rB, 16 * kk + 2 * q),
                                    f2(S0s, rA, 16 * kk + 2 * q + 8), f2(S0s, rB, 16 * kk + 2 * q + 8));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tt = 8 * nt + g;
                mma3(sa[nt], sf, make_b(f2(ap, tt, 16 * kk + 2 * q), f2(ap, tt, 16 * kk + 2 * q + 8)));
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int n = 16 + 8 * nt + g;
            mma3(sa[nt], vA,
                 make_b(make_float2(QM[(2 * q) * QS + n], QM[(2 * q + 1) * QS + n]),
                        make_float2(QM[(2 * q + 8) * QS + n], QM[(2 * q + 9) * QS + n])));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t = 8 * nt + 2 * q;
            SAt[t * SP + rA] = sa[nt][0];
            SAt[(t + 1) * SP + rA] = sa[nt][1];
            SAt[t * SP + rB] = sa[nt][2];
            SAt[(t + 1) * SP + rB] = sa[nt][3];
        }
        const AFrag saA = make_a(make_float2(sa[0][0], sa[0][1]), make_float2(sa[0][2], sa[0][3]),
                                 make_float2(sa[1][0], sa[1][1]), make_float2(sa[1][2], sa[1][3]));
        __syncthreads();  // A' (aliased by DSA) fully read

        // the dw running sum starts at diag(dsT^T sT): sT from the last chunk's start state
        if (last && p.dsT) {
            float ST[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j0 = 8 * nt + 2 * q;
                const float2 x = f2(S0s, rA, j0), z = f2(S0s, rB, j0);
                const float d0 = dd[(C - 1) * SP + j0], d1 = dd[(C - 1) * SP + j0 + 1];
                ST[nt][0] = x.x * d0; ST[nt][1] = x.y * d1; ST[nt][2] = z.x * d0; ST[nt][3] = z.y * d1;
                const int jn = 8 * nt + g;
                const float dcn = dd[(C - 1) * SP + jn];
                const BFrag bb = make_b(make_float2(bt[(2 * q) * SP + jn] * dcn, bt[(2 * q + 1) * SP + jn] * dcn),
                                        make_float2(bt[(2 * q + 8) * SP + jn] * dcn, bt[(2 * q + 9) * SP + jn] * dcn));
                const BFrag kb = make_b(make_float2(kt[(2 * q) * SP + jn] * dcn, kt[(2 * q + 1) * SP + jn] * dcn),
                                        make_float2(kt[(2 * q + 8) * SP + jn] * dcn, kt[(2 * q + 9) * SP + jn] * dcn));
                mma3(ST[nt], saA, bb);
                mma3(ST[nt], vA, kb);
                // column partials dsT o sT over this lane's rows, then over the warp's 16 rows
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float s = rows_sum(__fmaf_rn(Gh[nt][e], ST[nt][e], __fmul_rn(Gh[nt][2 + e], ST[nt][2 + e])));
                    if (g == 0) red_start[warp * 64 + j0 + e] = s;
                }
            }
            __syncthreads();
            carryA = red_start[rA] + red_start[64 + rA] + red_start[128 + rA] + red_start[192 + rA];
            carryB = red_start[rB] + red_start[64 + rB] + red_start[128 + rB] + red_start[192 + rB];
            __syncthreads();
        }

        // ---------------- G2: [DV | DSA] = G [K' | B'] + DY [Q'^T | (W Q_b)^T]
        float dvs[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag gf = a_from_acc(Gh, kk);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n = 8 * nt + g;
                mma3(dvs[nt], gf, make_b(f2(KB, n, 16 * kk + 2 * q), f2(KB, n, 16 * kk + 2 * q + 8)));
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int n = 8 * nt + g;
            mma3(dvs[nt], dyA,
                 make_b(*reinterpret_cast<const float2 *>(QQ + n * QQS + 2 * q),
                        *reinterpret_cast<const float2 *>(QQ + n * QQS + 2 * q + 8)));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {  // dv -> global (only real tokens)
            const int t = 8 * nt + 2 * q;
            if (t < nv) {
                p.dv[base0 + (size_t)(t0 + t) * tstride + rA] = dvs[nt][0];
                p.dv[base0 + (size_t)(t0 + t) * tstride + rB] = dvs[nt][2];
            }
            if (t + 1 < nv) {
                p.dv[base0 + (size_t)(t0 + t + 1) * tstride + rA] = dvs[nt][1];
                p.dv[base0 + (size_t)(t0 + t + 1) * tstride + rB] = dvs[nt][3];
            }
            DSt[t * SP + rA] = dvs[nt + 2][0];
            DSt[(t + 1) * SP + rA] = dvs[nt + 2][1];
            DSt[t * SP + rB] = dvs[nt + 2][2];
            DSt[(t + 1) * SP + rB] = dvs[nt + 2][3];
        }
        const AFrag dsA = make_a(make_float2(dvs[2][0], dvs[2][1]), make_float2(dvs[2][2], dvs[2][3]),
                                 make_float2(dvs[3][0], dvs[3][1]), make_float2(dvs[3][2], dvs[3][3]));
        __syncthreads();

        // ---------------- Gam = [SA | V]^T [DY | DSA] (32x32, over the 64 value rows)
        {
            const int mt = warp >> 1;
            const float *As = mt ? vt : SAt;
            float acc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const AFrag af = make_a(f2(As, g, 16 * kk + 2 * q), f2(As, g + 8, 16 * kk + 2 * q),
                                        f2(As, g, 16 * kk + 2 * q + 8), f2(As, g + 8, 16 * kk + 2 * q + 8));
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * (warp & 1) + u;
                    const float *Bs = nt < 2 ? dys : DSt;
                    const int tt = 8 * (nt & 1) + g;
                    mma3(acc[u], af, make_b(f2(Bs, tt, 16 * kk + 2 * q), f2(Bs, tt, 16 * kk + 2 * q + 8)));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int col = 8 * (2 * (warp & 1) + u) + 2 * q, row = 16 * mt + g;
                Gm[row * GS + col] = acc[u][0];
                Gm[row * GS + col + 1] = acc[u][1];
                Gm[(row + 8) * GS + col] = acc[u][2];
                Gm[(row + 8) * GS + col + 1] = acc[u][3];
            }
        }
        __syncthreads();

        // ---------------- G3: [DR | DA] (rows = key index j = rA/rB)
        float x3[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int i0 = 16 * kk + 2 * q;
            const AFrag sT = make_a(make_float2(S0s[i0 * SP + rA], S0s[(i0 + 1) * SP + rA]),
                                    make_float2(S0s[i0 * SP + rB], S0s[(i0 + 1) * SP + rB]),
                                    make_float2(S0s[(i0 + 8) * SP + rA], S0s[(i0 + 9) * SP + rA]),
                                    make_float2(S0s[(i0 + 8) * SP + rB], S0s[(i0 + 9) * SP + rB]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const float *Bs = nt < 2 ? dys : DSt;
                const int tt = 8 * (nt & 1) + g;
                mma3(x3[nt], sT, make_b(f2(Bs, tt, i0), f2(Bs, tt, i0 + 8)));
            }
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {  // [B~ | K~] mask(Gam): k-tile 0 pairs b~_s with sa rows, 1 k~_s with v rows
            const float *As = kk ? kt : bt;
            const AFrag af = make_a(make_float2(As[(2 * q) * SP + rA], As[(2 * q + 1) * SP + rA]),
                                    make_float2(As[(2 * q) * SP + rB], As[(2 * q + 1) * SP + rB]),
                                    make_float2(As[(2 * q + 8) * SP + rA], As[(2 * q + 9) * SP + rA]),
                                    make_float2(As[(2 * q + 8) * SP + rB], As[(2 * q + 9) * SP + rB]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n = 8 * nt + g, t = n & 15;
                const bool strict = nt >= 2;  // dsa columns: s < t ; dy columns: s <= t
                float e[4];
                const int s4[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int s = s4[m];
                    const bool keep = strict ? (s < t) : (s <= t);
                    e[m] = keep ? Gm[(16 * kk + s) * GS + n] : 0.f;
                }
                mma3(x3[nt], af, make_b(make_float2(e[0], e[1]), make_float2(e[2], e[3])));
            }
        }
        __syncthreads();  // S_0 and dy no longer read: fetch the previous chunk's
        if (c > 0) {
            stage_rows<NT>(dys, p.dy + base0 + (size_t)(t0 - C) * tstride, tstride, C, C);
            stage_rows<NT>(S0s, p.ckpt_in + ((size_t)bh * p.nck + c - 1) * 64 * 64, 64, 64, 64);
        }
        cp_async_commit();

        // ---------------- G4: [DK | DB] (rows = key index)
        float x4[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int i0 = 16 * kk + 2 * q;
            const AFrag gT = make_a(make_float2(Gds[i0 * SP + rA], Gds[(i0 + 1) * SP + rA]),
                                    make_float2(Gds[i0 * SP + rB], Gds[(i0 + 1) * SP + rB]),
                                    make_float2(Gds[(i0 + 8) * SP + rA], Gds[(i0 + 9) * SP + rA]),
                                    make_float2(Gds[(i0 + 8) * SP + rB], Gds[(i0 + 9) * SP + rB]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const float *Bs = nt < 2 ? vt : SAt;
                const int tt = 8 * (nt & 1) + g;
                mma3(x4[nt], gT, make_b(f2(Bs, tt, i0), f2(Bs, tt, i0 + 8)));
            }
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {  // [R^ | A^] mask(Gam^T): k-tile 0 pairs r^_s with dy_s, 1 a^_s with dsa_s
            const float *As = kk ? ah : rh;
            const AFrag af = make_a(make_float2(As[(2 * q) * SP + rA], As[(2 * q + 1) * SP + rA]),
                                    make_float2(As[(2 * q) * SP + rB], As[(2 * q + 1) * SP + rB]),
                                    make_float2(As[(2 * q + 8) * SP + rA], As[(2 * q + 9) * SP + rA]),
                                    make_float2(As[(2 * q + 8) * SP + rB], As[(2 * q + 9) * SP + rB]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n = 8 * nt + g, t = n & 15;
                const int grow = nt < 2 ? 16 + t : t;  // v_t rows (16..31) for dk, sa_t rows (0..15) for db
                float e[4];
                const int s4[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int s = s4[m];
                    const bool keep = kk ? (s > t) : (s >= t);
                    e[m] = keep ? Gm[grow * GS + 16 * kk + s] : 0.f;
                }
                mma3(x4[nt], af, make_b(make_float2(e[0], e[1]), make_float2(e[2], e[3])));
            }
        }

        // ---------------- outputs of the key-indexed gradients and the dw running sum
        {
            // z_t = r^ o X3_r + a^ o X3_a - b~ o X4_b - k~ o X4_k ; e_t = a^ o X3_a
            float zz[2][4], ee[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int row = m < 2 ? rA : rB;
                    const int t = 8 * nt + 2 * q + (m & 1);
                    const float d = dd[t * SP + row];
                    const float dp = t ? dd[(t - 1) * SP + row] : 1.f;
                    const float inv = __frcp_rn(d);
                    const float xr = x3[nt][m], xa = x3[nt + 2][m], xk = x4[nt][m], xb = x4[nt + 2][m];
                    ee[nt][m] = ah[t * SP + row] * xa;
                    zz[nt][m] = rh[t * SP + row] * xr + ee[nt][m] - bt[t * SP + row] * xb - kt[t * SP + row] * xk;
                    if (t < nv) {
                        const size_t o = base0 + (size_t)(t0 + t) * tstride + row;
                        p.dr[o] = d * xr;
                        p.da[o] = dp * xa;
                        p.dk[o] = inv * xk;
                        p.db[o] = inv * xb;
                    }
                }
            // reverse running sums over t per key row (rows rA: m = 0,1 ; rB: m = 2,3)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float carry = hr ? carryB : carryA;
                const int row = hr ? rB : rA;
                const float P0 = zz[0][2 * hr] + zz[0][2 * hr + 1];
                const float P1 = zz[1][2 * hr] + zz[1][2 * hr + 1];
                float s0 = P0, s1 = P1;  // inclusive suffix sums over q within the quad
                float y;
                y = __shfl_down_sync(kFull, s0, 1, 4); if (q < 3) s0 += y;
                y = __shfl_down_sync(kFull, s0, 2, 4); if (q < 2) s0 += y;
                y = __shfl_down_sync(kFull, s1, 1, 4); if (q < 3) s1 += y;
                y = __shfl_down_sync(kFull, s1, 2, 4); if (q < 2) s1 += y;
                const float upper = __shfl_sync(kFull, s1, 0, 4);
                const float lowAfter = s0 - P0, upAfter = s1 - P1;
                const float S9 = zz[1][2 * hr + 1] + upAfter + carry;   // t = 9 + 2q
                const float S8 = zz[1][2 * hr] + S9;                    // t = 8 + 2q
                const float S1 = zz[0][2 * hr + 1] + lowAfter + upper + carry;  // t = 2q + 1
                const float S0v = zz[0][2 * hr] + S1;                   // t = 2q
                const float Sv[4] = {S0v, S1, S8, S9};
                const int tv[4] = {2 * q, 2 * q + 1, 8 + 2 * q, 9 + 2 * q};
                const float ev[4] = {ee[0][2 * hr], ee[0][2 * hr + 1], ee[1][2 * hr], ee[1][2 * hr + 1]};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = tv[m];
                    if (t < nv) {
                        const float d = dd[t * SP + row];
                        const float dp = t ? dd[(t - 1) * SP + row] : 1.f;
                        p.dw[base0 + (size_t)(t0 + t) * tstride + row] = (Sv[m] - ev[m]) * (dp * __frcp_rn(d));
                    }
                }
                const float total = __shfl_sync(kFull, S0v, 0, 4);  // sum over the whole chunk + carry
                if (hr) carryB = total; else carryA = total;
            }
        }

        // ---------------- G5: G_prev = Gd + [DY | DSA] [R^ | A^]^T  (rows = value index)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int jn = 8 * nt + g;
            const BFrag br = make_b(make_float2(rh[(2 * q) * SP + jn], rh[(2 * q + 1) * SP + jn]),
                                    make_float2(rh[(2 * q + 8) * SP + jn], rh[(2 * q + 9) * SP + jn]));
            const BFrag ba = make_b(make_float2(ah[(2 * q) * SP + jn], ah[(2 * q + 1) * SP + jn]),
                                    make_float2(ah[(2 * q + 8) * SP + jn], ah[(2 * q + 9) * SP + jn]));
            mma3(Gd[nt], dyA, br);
            mma3(Gd[nt], dsA, ba);
#pragma unroll
            for (int m = 0; m < 4; ++m) Gh[nt][m] = Gd[nt][m];
        }
        __syncthreads();
    }
    cp_async_wait_all();
    if (p.ds0) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<float2 *>(p.ds0 + sbase + rA * 64 + 8 * nt + 2 * q) = make_float2(Gh[nt][0], Gh[nt][1]);
            *reinterpret_cast<float2 *>(p.ds0 + sbase + rB * 64 + 8 * nt + 2 * q) = make_float2(Gh[nt][2], Gh[nt][3]);
        }
    }
}

}  // namespace

bool backward_chunk_supported(const SeqArgs &p) { return p.L == C; }

cudaError_t launch_backward_chunk(const SeqArgs &p, cudaStream_t st) {
    const int grid = p.B * p.H;
    cudaError_t e;
    if (p.dtype == 1) {
        const size_t sm = bwd_smem_bytes<__nv_bfloat16>();
        if ((e = cudaFuncSetAttribute(wkv7_bwd_chunk_kernel<__nv_bfloat16>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) != cudaSuccess)
            return e;
        wkv7_bwd_chunk_kernel<__nv_bfloat16><<<grid, NT, sm, st>>>(p);
    } else {
        const size_t sm = bwd_smem_bytes<float>();
        if ((e = cudaFuncSetAttribute(wkv7_bwd_chunk_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)sm)) != cudaSuccess)
            return e;
        wkv7_bwd_chunk_kernel<float><<<grid, NT, sm, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace wkv7
