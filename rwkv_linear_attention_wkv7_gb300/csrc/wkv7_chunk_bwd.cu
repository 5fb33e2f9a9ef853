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
constexpr unsigned kFull = 0xffffffffu;

// Float offsets of the shared-memory carve-up (after the raw input block).
constexpr int O_DY = 0;                   // dy       [C][SP]
constexpr int O_S0 = O_DY + C * SP;       // S_0      [64][SP]
constexpr int O_GD = O_S0 + 64 * SP;      // G d_C    [64][SP]  (exact path: S_{t-1})
constexpr int O_DD = O_GD + 64 * SP;      // d        [C][SP]
constexpr int O_G = O_DD + C * SP;        // Gram, then Gam [32][GS]
constexpr int O_W = O_G + C * SP;         // W [C][WS]
constexpr int O_QM = O_W + C * WS;        // M_k' in columns 16..31 [C][QS]
constexpr int O_SAT = O_QM + C * QS;      // SA (token-major) [C][SP]
constexpr int O_DST = O_SAT + C * SP;     // DSA (token-major) [C][SP]; dw start scratch
constexpr int O_X = O_DST + C * SP;       // u32 x 4096: G1/G2 operands, then [DY|DSA], [V|SA]; exact-path scratch
constexpr int O_B5 = O_X + 4096;          // u32 x 2048: B of G_prev's product
constexpr int O_GM = O_B5 + 2048;         // u32 x 2048: masked Gam blocks
constexpr int kFloats = O_GM + 2048;
static_assert(32 * GS <= C * SP, "Gam must fit its slot");
static_assert(5 * 4 * 64 <= 4096, "exact-path scratch must fit region X");
static_assert(O_X % 4 == 0 && O_B5 % 4 == 0 && O_GM % 4 == 0, "16-byte fragment buffers");

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


__device__ __forceinline__ uint4 pack_b(float x0, float x1, float x8, float x9) {
    const Frag2 a = split2(x0, x1), b = split2(x8, x9);
    return make_uint4(a.hi, b.hi, a.lo, b.lo);
}
__device__ __forceinline__ BFrag ld_b(const uint32_t *buf, int idx) {
    const uint4 u = reinterpret_cast<const uint4 *>(buf)[idx];
    BFrag f;
    f.hi[0] = u.x; f.hi[1] = u.y; f.lo[0] = u.z; f.lo[1] = u.w;
    return f;
}
// A fragment (16 rows x 16 k) assembled from the B fragments of the two
// n-tiles that hold those rows (same element pairs, other register order).
__device__ __forceinline__ AFrag a_from_b(const uint32_t *buf, int idx_rows0_7, int idx_rows8_15) {
    const uint4 u = reinterpret_cast<const uint4 *>(buf)[idx_rows0_7];
    const uint4 v = reinterpret_cast<const uint4 *>(buf)[idx_rows8_15];
    AFrag f;
    f.hi[0] = u.x; f.hi[1] = v.x; f.hi[2] = u.y; f.hi[3] = v.y;
    f.lo[0] = u.z; f.lo[1] = v.z; f.lo[2] = u.w; f.lo[3] = v.w;
    return f;
}
__device__ __forceinline__ void st_b_half(uint32_t *buf, int idx, int half, const Frag2 &f) {
    buf[idx * 4 + half] = f.hi;
    buf[idx * 4 + 2 + half] = f.lo;
}

template <typename E>
__global__ void __launch_bounds__(NT, 2) wkv7_bwd_chunk_kernel(SeqArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);
    float *F = reinterpret_cast<float *>(smem + raw_bytes<E>());
    float *dys = F + O_DY, *S0s = F + O_S0, *Gds = F + O_GD, *dd = F + O_DD, *Gm = F + O_G, *Wm = F + O_W;
    float *QM = F + O_QM, *SAt = F + O_SAT, *DSt = F + O_DST;
    uint32_t *X = reinterpret_cast<uint32_t *>(F + O_X);
    uint32_t *B1 = X, *B1V = X + 1024, *B2 = X + 1280, *B2D = X + 3328;  // per-chunk operands
    uint32_t *DYDS = X, *VSA = X + 2048;                                  // after G1/G2
    uint32_t *B5 = reinterpret_cast<uint32_t *>(F + O_B5);
    uint32_t *GM3 = reinterpret_cast<uint32_t *>(F + O_GM), *GM4 = GM3 + 1024;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int bh = blockIdx.x, bi = bh / p.H, h = bh % p.H;
    const size_t tstride = (size_t)p.H * 64;
    const size_t base0 = ((size_t)bi * p.T * p.H + h) * 64;
    const size_t sbase = (size_t)bh * 64 * 64;
    const int rA = warp * 16 + g, rB = rA + 8;  // value rows (row-owned products) / key rows (G3, G4)

    auto a_hat = [&](int t, int j) { return ld_raw(raw, VA, t, j) * (t ? dd[(t - 1) * SP + j] : 1.f); };
    auto r_hat = [&](int t, int j) { return ld_raw(raw, VR, t, j) * dd[t * SP + j]; };
    auto b_til = [&](int t, int j) { return ld_raw(raw, VB, t, j) * rcp_approx(dd[t * SP + j]); };
    auto k_til = [&](int t, int j) { return ld_raw(raw, VK, t, j) * rcp_approx(dd[t * SP + j]); };
    // pairs (j, j + 1), j even: one load each for the input and the decay
    auto d2 = [&](int t, int j) { return *reinterpret_cast<const float2 *>(dd + t * SP + j); };
    auto a_hat2 = [&](int t, int j) {
        const float2 x = ld_raw2(raw, VA, t, j);
        const float2 d = t ? d2(t - 1, j) : make_float2(1.f, 1.f);
        return make_float2(x.x * d.x, x.y * d.y);
    };
    auto r_hat2 = [&](int t, int j) {
        const float2 x = ld_raw2(raw, VR, t, j), d = d2(t, j);
        return make_float2(x.x * d.x, x.y * d.y);
    };
    auto bk_til2 = [&](int vec, int t, int j) {
        const float2 x = ld_raw2(raw, vec, t, j), d = d2(t, j);
        return make_float2(x.x * rcp_approx(d.x), x.y * rcp_approx(d.y));
    };

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
    {
        const int c = nchunks - 1, t0 = c * C, nv = min(C, p.T - t0);
        stage<E, 6, NT>(raw, src, base0 + (size_t)t0 * tstride, tstride, nv);
        stage_rows<NT>(dys, p.dy + base0 + (size_t)t0 * tstride, tstride, C, nv);
        stage_rows<NT>(S0s, p.ckpt_in + ((size_t)bh * p.nck + c) * 64 * 64, 64, 64, 64);
        cp_async_commit();
    }

    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        const bool last = c == nchunks - 1;
        cp_async_wait_all();
        __syncthreads();

        const bool exact = __syncthreads_or(prep_decay(raw, dd, nv));
        if (exact) {
            bwd_chunk_exact<E>(raw, dys, S0s, Gds, reinterpret_cast<float *>(X), Gh, nv, p, base0, tstride, t0,
                               carryA, carryB);
            __syncthreads();
            if (c > 0) {
                stage<E, 6, NT>(raw, src, base0 + (size_t)(t0 - C) * tstride, tstride, C);
                stage_rows<NT>(dys, p.dy + base0 + (size_t)(t0 - C) * tstride, tstride, C, C);
                stage_rows<NT>(S0s, p.ckpt_in + ((size_t)bh * p.nck + c - 1) * 64 * 64, 64, 64, 64);
            }
            cp_async_commit();
            continue;
        }
        const float *dC = dd + (C - 1) * SP;

        // ================= per-chunk operands (no state involved)
        // Gram [B~; K~] [A^; R^]^T on the fly: warp -> m-tile (b~ | k~), two n-tiles (a^ | r^)
        {
            const int mt = warp >> 1;
            float acc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int j0 = 16 * kk + 2 * q;
                const int av = mt ? VK : VB;
                const AFrag af = make_a(bk_til2(av, g, j0), bk_til2(av, g + 8, j0), bk_til2(av, g, j0 + 8),
                                        bk_til2(av, g + 8, j0 + 8));
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * (warp & 1) + u;
                    const int tt = 8 * (nt & 1) + g;
                    const BFrag bf = nt < 2 ? make_b(a_hat2(tt, j0), a_hat2(tt, j0 + 8)) : make_b(r_hat2(tt, j0), r_hat2(tt, j0 + 8));
                    mma3(acc[u], af, bf);
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
        // B fragments of G_prev's product [DY | DSA] [R^ | A^]^T: B[k = token][n = key column]
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int f = tid + NT * m;  // 512 fragments: kt = f >> 8 (0: r^, 1: a^), nt = (f >> 5) & 7
            const int kt = f >> 8, nt = (f >> 5) & 7, ln = f & 31, gg = ln >> 2, qq = ln & 3, j = 8 * nt + gg;
            float x[4];
            const int s4[4] = {2 * qq, 2 * qq + 1, 2 * qq + 8, 2 * qq + 9};
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = kt ? a_hat(s4[e], j) : r_hat(s4[e], j);
            reinterpret_cast<uint4 *>(B5)[f] = pack_b(x[0], x[1], x[2], x[3]);
        }
        // G diag(d_C) for Gd^T (rows = value index)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int j0 = 8 * nt + 2 * q;
            const float2 dc = *reinterpret_cast<const float2 *>(dC + j0);
            *reinterpret_cast<float2 *>(Gds + rA * SP + j0) = make_float2(Gh[nt][0] * dc.x, Gh[nt][1] * dc.y);
            *reinterpret_cast<float2 *>(Gds + rB * SP + j0) = make_float2(Gh[nt][2] * dc.x, Gh[nt][3] * dc.y);
        }
        __syncthreads();
        prep_inverse(Gm, Wm);
        __syncthreads();

        // W^T as an A operand: wt[t][s] = W[s][t]
        const AFrag wt = make_a(make_float2(Wm[(2 * q) * WS + g], Wm[(2 * q + 1) * WS + g]),
                                make_float2(Wm[(2 * q) * WS + g + 8], Wm[(2 * q + 1) * WS + g + 8]),
                                make_float2(Wm[(2 * q + 8) * WS + g], Wm[(2 * q + 9) * WS + g]),
                                make_float2(Wm[(2 * q + 8) * WS + g + 8], Wm[(2 * q + 9) * WS + g + 8]));
        // A' = W^T-weighted A^ (M = token, N = key; warp w owns keys 16w..16w+15) -> B of G1
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int jn = 16 * warp + 8 * u + g;
            float ca[4] = {0.f, 0.f, 0.f, 0.f};
            mma3(ca, wt, make_b(make_float2(a_hat(2 * q, jn), a_hat(2 * q + 1, jn)),
                                make_float2(a_hat(2 * q + 8, jn), a_hat(2 * q + 9, jn))));
            // G1 B layout: [kt = warp][nt = token half][lane], register half u
            st_b_half(B1, (warp * 2 + 0) * 32 + lane, u, split2(ca[0], ca[1]));
            st_b_half(B1, (warp * 2 + 1) * 32 + lane, u, split2(ca[2], ca[3]));
        }
        if (warp == 0) {  // M_k' = M_k W, Q' = Q_k + M_k' Q_b, Q_b' = W Q_b (all 16 x 16)
            auto mk = [&](int s, int u) { return u > s ? Gm[(16 + s) * GS + u] : 0.f; };
            auto qbv = [&](int u, int t) { return u <= t ? Gm[u * GS + 16 + t] : 0.f; };
            auto qkv = [&](int s, int t) { return s <= t ? Gm[(16 + s) * GS + 16 + t] : 0.f; };
            const AFrag am = make_a(make_float2(mk(g, 2 * q), mk(g, 2 * q + 1)), make_float2(mk(g + 8, 2 * q), mk(g + 8, 2 * q + 1)),
                                    make_float2(mk(g, 2 * q + 8), mk(g, 2 * q + 9)),
                                    make_float2(mk(g + 8, 2 * q + 8), mk(g + 8, 2 * q + 9)));
            const AFrag wa = make_a(make_float2(Wm[g * WS + 2 * q], Wm[g * WS + 2 * q + 1]),
                                    make_float2(Wm[(g + 8) * WS + 2 * q], Wm[(g + 8) * WS + 2 * q + 1]),
                                    make_float2(Wm[g * WS + 2 * q + 8], Wm[g * WS + 2 * q + 9]),
                                    make_float2(Wm[(g + 8) * WS + 2 * q + 8], Wm[(g + 8) * WS + 2 * q + 9]));
            float cm[2][4] = {}, cb[2][4] = {};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t = 8 * nt + g;
                mma3(cm[nt], am, make_b(make_float2(Wm[(2 * q) * WS + t], Wm[(2 * q + 1) * WS + t]),
                                        make_float2(Wm[(2 * q + 8) * WS + t], Wm[(2 * q + 9) * WS + t])));
                mma3(cb[nt], wa, make_b(make_float2(qbv(2 * q, t), qbv(2 * q + 1, t)),
                                        make_float2(qbv(2 * q + 8, t), qbv(2 * q + 9, t))));
            }
            const AFrag amp = make_a(make_float2(cm[0][0], cm[0][1]), make_float2(cm[0][2], cm[0][3]),
                                     make_float2(cm[1][0], cm[1][1]), make_float2(cm[1][2], cm[1][3]));
            float cq[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tc = 8 * nt + 2 * q, t = 8 * nt + g;
                cq[nt][0] = qkv(g, tc); cq[nt][1] = qkv(g, tc + 1); cq[nt][2] = qkv(g + 8, tc); cq[nt][3] = qkv(g + 8, tc + 1);
                mma3(cq[nt], amp, make_b(make_float2(qbv(2 * q, t), qbv(2 * q + 1, t)),
                                         make_float2(qbv(2 * q + 8, t), qbv(2 * q + 9, t))));
            }
            // DY-side B of G2: B[k = s][n] = Q'[n][s] (n < 16), (W Q_b)[n - 16][s]; C rows of Q' / W Q_b are n
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {  // column half nt of the C tile = register half of the B fragment
                st_b_half(B2D, 0 * 32 + lane, nt, split2(cq[nt][0], cq[nt][1]));
                st_b_half(B2D, 1 * 32 + lane, nt, split2(cq[nt][2], cq[nt][3]));
                st_b_half(B2D, 2 * 32 + lane, nt, split2(cb[nt][0], cb[nt][1]));
                st_b_half(B2D, 3 * 32 + lane, nt, split2(cb[nt][2], cb[nt][3]));
                const int tc = 8 * nt + 2 * q;
                QM[g * QS + 16 + tc] = cm[nt][0]; QM[g * QS + 16 + tc + 1] = cm[nt][1];
                QM[(g + 8) * QS + 16 + tc] = cm[nt][2]; QM[(g + 8) * QS + 16 + tc + 1] = cm[nt][3];
            }
            __syncwarp();
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {  // V-side B of G1: B[k = s][n = t] = M_k'[s][t]
                const int n = 16 + 8 * nt + g;
                reinterpret_cast<uint4 *>(B1V)[nt * 32 + lane] =
                    pack_b(QM[(2 * q) * QS + n], QM[(2 * q + 1) * QS + n], QM[(2 * q + 8) * QS + n], QM[(2 * q + 9) * QS + n]);
            }
        }
        __syncthreads();
        // K' = d_C o (K~ + M_k' B~) and B' = d_C o (W B~)  (M = token, N = key) -> B of G2
        {
            auto mkp = [&](int t, int s) { return QM[t * QS + 16 + s]; };
            const AFrag amk = make_a(make_float2(mkp(g, 2 * q), mkp(g, 2 * q + 1)), make_float2(mkp(g + 8, 2 * q), mkp(g + 8, 2 * q + 1)),
                                     make_float2(mkp(g, 2 * q + 8), mkp(g, 2 * q + 9)),
                                     make_float2(mkp(g + 8, 2 * q + 8), mkp(g + 8, 2 * q + 9)));
            const AFrag awn = make_a(make_float2(Wm[g * WS + 2 * q], Wm[g * WS + 2 * q + 1]),
                                     make_float2(Wm[(g + 8) * WS + 2 * q], Wm[(g + 8) * WS + 2 * q + 1]),
                                     make_float2(Wm[g * WS + 2 * q + 8], Wm[g * WS + 2 * q + 9]),
                                     make_float2(Wm[(g + 8) * WS + 2 * q + 8], Wm[(g + 8) * WS + 2 * q + 9]));
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int jn = 16 * warp + 8 * u + g, jc = 16 * warp + 8 * u + 2 * q;
                const BFrag bb = make_b(make_float2(b_til(2 * q, jn), b_til(2 * q + 1, jn)),
                                        make_float2(b_til(2 * q + 8, jn), b_til(2 * q + 9, jn)));
                float ck[4] = {k_til(g, jc), k_til(g, jc + 1), k_til(g + 8, jc), k_til(g + 8, jc + 1)};
                float cb2[4] = {0.f, 0.f, 0.f, 0.f};
                mma3(ck, amk, bb);
                mma3(cb2, awn, bb);
                const float2 dc = *reinterpret_cast<const float2 *>(dC + jc);
                ck[0] *= dc.x; ck[1] *= dc.y; ck[2] *= dc.x; ck[3] *= dc.y;
                cb2[0] *= dc.x; cb2[1] *= dc.y; cb2[2] *= dc.x; cb2[3] *= dc.y;
                // G2 B layout: [kt = warp][nt: 0,1 = K' token halves, 2,3 = B'][lane], register half u
                st_b_half(B2, (warp * 4 + 0) * 32 + lane, u, split2(ck[0], ck[1]));
                st_b_half(B2, (warp * 4 + 1) * 32 + lane, u, split2(ck[2], ck[3]));
                st_b_half(B2, (warp * 4 + 2) * 32 + lane, u, split2(cb2[0], cb2[1]));
                st_b_half(B2, (warp * 4 + 3) * 32 + lane, u, split2(cb2[2], cb2[3]));
            }
        }
        __syncthreads();

        // ================= state-dependent products
        const AFrag vA = make_a(make_float2(ld_raw(raw, VV, 2 * q, rA), ld_raw(raw, VV, 2 * q + 1, rA)),
                                make_float2(ld_raw(raw, VV, 2 * q, rB), ld_raw(raw, VV, 2 * q + 1, rB)),
                                make_float2(ld_raw(raw, VV, 2 * q + 8, rA), ld_raw(raw, VV, 2 * q + 9, rA)),
                                make_float2(ld_raw(raw, VV, 2 * q + 8, rB), ld_raw(raw, VV, 2 * q + 9, rB)));
        const AFrag dyA = make_a(make_float2(dys[(2 * q) * SP + rA], dys[(2 * q + 1) * SP + rA]),
                                 make_float2(dys[(2 * q) * SP + rB], dys[(2 * q + 1) * SP + rB]),
                                 make_float2(dys[(2 * q + 8) * SP + rA], dys[(2 * q + 9) * SP + rA]),
                                 make_float2(dys[(2 * q + 8) * SP + rB], dys[(2 * q + 9) * SP + rB]));
        // G1: SA = S_0 A' + V M_k'  (rows = value index)
        float sa[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag sf = make_a(f2(S0s, rA, 16 * kk + 2 * q), f2(S0s, rB, 16 * kk + 2 * q),
                                    f2(S0s, rA, 16 * kk + 2 * q + 8), f2(S0s, rB, 16 * kk + 2 * q + 8));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma3(sa[nt], sf, ld_b(B1, (kk * 2 + nt) * 32 + lane));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma3(sa[nt], vA, ld_b(B1V, nt * 32 + lane));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t = 8 * nt + 2 * q;
            SAt[t * SP + rA] = sa[nt][0];
            SAt[(t + 1) * SP + rA] = sa[nt][1];
            SAt[t * SP + rB] = sa[nt][2];
            SAt[(t + 1) * SP + rB] = sa[nt][3];
        }

        // the dw running sum starts at diag(dsT^T sT): sT from the last chunk's start state
        if (last && p.dsT) {
            const AFrag saA = make_a(make_float2(sa[0][0], sa[0][1]), make_float2(sa[0][2], sa[0][3]),
                                     make_float2(sa[1][0], sa[1][1]), make_float2(sa[1][2], sa[1][3]));
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j0 = 8 * nt + 2 * q;
                const float2 x = f2(S0s, rA, j0), z = f2(S0s, rB, j0);
                const float2 dc = *reinterpret_cast<const float2 *>(dC + j0);
                float ST[4] = {x.x * dc.x, x.y * dc.y, z.x * dc.x, z.y * dc.y};
                const int jn = 8 * nt + g;
                const float dcn = dC[jn];
                const BFrag bb = make_b(make_float2(b_til(2 * q, jn) * dcn, b_til(2 * q + 1, jn) * dcn),
                                        make_float2(b_til(2 * q + 8, jn) * dcn, b_til(2 * q + 9, jn) * dcn));
                const BFrag kb = make_b(make_float2(k_til(2 * q, jn) * dcn, k_til(2 * q + 1, jn) * dcn),
                                        make_float2(k_til(2 * q + 8, jn) * dcn, k_til(2 * q + 9, jn) * dcn));
                mma3(ST, saA, bb);
                mma3(ST, vA, kb);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float s = rows_sum(__fmaf_rn(Gh[nt][e], ST[e], __fmul_rn(Gh[nt][2 + e], ST[2 + e])));
                    if (g == 0) DSt[warp * 64 + j0 + e] = s;
                }
            }
            __syncthreads();
            carryA = DSt[rA] + DSt[64 + rA] + DSt[128 + rA] + DSt[192 + rA];
            carryB = DSt[rB] + DSt[64 + rB] + DSt[128 + rB] + DSt[192 + rB];
            __syncthreads();
        }

        // G2: [DV | DSA] = G [K' | B'] + DY [Q'^T | (W Q_b)^T]
        float dvs[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag gf = a_from_acc(Gh, kk);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma3(dvs[nt], gf, ld_b(B2, (kk * 4 + nt) * 32 + lane));
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma3(dvs[nt], dyA, ld_b(B2D, nt * 32 + lane));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
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

        // [DY | DSA] and [V | SA] as B operands over the value rows: B[k = i][n = token]
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int f = tid + NT * m;  // 1024 fragments: which = f >> 9, kt = (f >> 7) & 3, nt = (f >> 5) & 3
            const int which = f >> 9, kt = (f >> 7) & 3, nt = (f >> 5) & 3, ln = f & 31, gg = ln >> 2, qq = ln & 3;
            const int t = 8 * (nt & 1) + gg, i0 = 16 * kt + 2 * qq;
            float x0, x1, x8, x9;
            if (which == 0) {
                const float *s_ = nt < 2 ? dys : DSt;
                const float2 a = f2(s_, t, i0), b = f2(s_, t, i0 + 8);
                x0 = a.x; x1 = a.y; x8 = b.x; x9 = b.y;
            } else if (nt < 2) {
                const float2 a = ld_raw2(raw, VV, t, i0), b = ld_raw2(raw, VV, t, i0 + 8);
                x0 = a.x; x1 = a.y; x8 = b.x; x9 = b.y;
            } else {
                const float2 a = f2(SAt, t, i0), b = f2(SAt, t, i0 + 8);
                x0 = a.x; x1 = a.y; x8 = b.x; x9 = b.y;
            }
            reinterpret_cast<uint4 *>(which ? VSA : DYDS)[(kt * 4 + nt) * 32 + ln] = pack_b(x0, x1, x8, x9);
        }
        __syncthreads();

        // Gam = [SA | V]^T [DY | DSA] (32 x 32): warp -> m-tile (SA rows | V rows), two n-tiles
        {
            const int mt = warp >> 1;
            float acc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int nb = mt ? 0 : 2;  // VSA n-tiles holding V (0,1) or SA (2,3)
                const AFrag af = a_from_b(VSA, (kk * 4 + nb) * 32 + lane, (kk * 4 + nb + 1) * 32 + lane);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * (warp & 1) + u;
                    mma3(acc[u], af, ld_b(DYDS, (kk * 4 + nt) * 32 + lane));
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
        // masked Gam blocks as B fragments: GM3 pairs (b~_s | k~_s) with (dy_t | dsa_t),
        // GM4 pairs (r^_s | a^_s) with (v_t | sa_t)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int f = tid + NT * m;  // 512: which = f >> 8, kt = (f >> 7) & 1, nt = (f >> 5) & 3
            const int which = f >> 8, kt = (f >> 7) & 1, nt = (f >> 5) & 3, ln = f & 31, gg = ln >> 2, qq = ln & 3;
            const int n = 8 * nt + gg, t = n & 15;
            const int s4[4] = {2 * qq, 2 * qq + 1, 2 * qq + 8, 2 * qq + 9};
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s = s4[e];
                if (which == 0) {
                    const bool keep = nt >= 2 ? (s < t) : (s <= t);
                    x[e] = keep ? Gm[(16 * kt + s) * GS + n] : 0.f;
                } else {
                    const int grow = nt < 2 ? 16 + t : t;
                    const bool keep = kt ? (s > t) : (s >= t);
                    x[e] = keep ? Gm[grow * GS + 16 * kt + s] : 0.f;
                }
            }
            reinterpret_cast<uint4 *>(which ? GM4 : GM3)[(kt * 4 + nt) * 32 + ln] = pack_b(x[0], x[1], x[2], x[3]);
        }
        __syncthreads();

        // G3: [DR | DA] (rows = key index j = rA / rB)
        float x3[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int i0 = 16 * kk + 2 * q;
            const AFrag sT = make_a(make_float2(S0s[i0 * SP + rA], S0s[(i0 + 1) * SP + rA]),
                                    make_float2(S0s[i0 * SP + rB], S0s[(i0 + 1) * SP + rB]),
                                    make_float2(S0s[(i0 + 8) * SP + rA], S0s[(i0 + 9) * SP + rA]),
                                    make_float2(S0s[(i0 + 8) * SP + rB], S0s[(i0 + 9) * SP + rB]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma3(x3[nt], sT, ld_b(DYDS, (kk * 4 + nt) * 32 + lane));
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {  // [B~ | K~] (rows j, k = token)
            float x[8];
            const int s4[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = kk ? k_til(s4[e], rA) : b_til(s4[e], rA);
                x[2 * e + 1] = kk ? k_til(s4[e], rB) : b_til(s4[e], rB);
            }
            const AFrag af = make_a(make_float2(x[0], x[2]), make_float2(x[1], x[3]), make_float2(x[4], x[6]),
                                    make_float2(x[5], x[7]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma3(x3[nt], af, ld_b(GM3, (kk * 4 + nt) * 32 + lane));
        }
        __syncthreads();  // S_0 and dy no longer read: fetch the previous chunk's
        if (c > 0) {
            stage_rows<NT>(dys, p.dy + base0 + (size_t)(t0 - C) * tstride, tstride, C, C);
            stage_rows<NT>(S0s, p.ckpt_in + ((size_t)bh * p.nck + c - 1) * 64 * 64, 64, 64, 64);
        }
        cp_async_commit();

        // G4: [DK | DB] (rows = key index)
        float x4[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int i0 = 16 * kk + 2 * q;
            const AFrag gT = make_a(make_float2(Gds[i0 * SP + rA], Gds[(i0 + 1) * SP + rA]),
                                    make_float2(Gds[i0 * SP + rB], Gds[(i0 + 1) * SP + rB]),
                                    make_float2(Gds[(i0 + 8) * SP + rA], Gds[(i0 + 9) * SP + rA]),
                                    make_float2(Gds[(i0 + 8) * SP + rB], Gds[(i0 + 9) * SP + rB]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma3(x4[nt], gT, ld_b(VSA, (kk * 4 + nt) * 32 + lane));
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {  // [R^ | A^] (rows j, k = token)
            float x[8];
            const int s4[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = kk ? a_hat(s4[e], rA) : r_hat(s4[e], rA);
                x[2 * e + 1] = kk ? a_hat(s4[e], rB) : r_hat(s4[e], rB);
            }
            const AFrag af = make_a(make_float2(x[0], x[2]), make_float2(x[1], x[3]), make_float2(x[4], x[6]),
                                    make_float2(x[5], x[7]));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma3(x4[nt], af, ld_b(GM4, (kk * 4 + nt) * 32 + lane));
        }

        // outputs of the key-indexed gradients and the dw running sum
        {
            float zz[2][4], ee[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int row = m < 2 ? rA : rB;
                    const int t = 8 * nt + 2 * q + (m & 1);
                    const float d = dd[t * SP + row];
                    const float dp = t ? dd[(t - 1) * SP + row] : 1.f;
                    const float inv = rcp_approx(d);
                    const float xr = x3[nt][m], xa = x3[nt + 2][m], xk = x4[nt][m], xb = x4[nt + 2][m];
                    const float rv = ld_raw(raw, VR, t, row), av = ld_raw(raw, VA, t, row);
                    const float bv = ld_raw(raw, VB, t, row), kv = ld_raw(raw, VK, t, row);
                    // r o dr = r^ o X3_r, a o da = a^ o X3_a, b o db = b~ o X4_b, k o dk = k~ o X4_k
                    ee[nt][m] = av * dp * xa;
                    zz[nt][m] = rv * d * xr + ee[nt][m] - bv * inv * xb - kv * inv * xk;
                    if (t < nv) {
                        const size_t o = base0 + (size_t)(t0 + t) * tstride + row;
                        p.dr[o] = d * xr;
                        p.da[o] = dp * xa;
                        p.dk[o] = inv * xk;
                        p.db[o] = inv * xb;
                    }
                }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float carry = hr ? carryB : carryA;
                const int row = hr ? rB : rA;
                const float P0 = zz[0][2 * hr] + zz[0][2 * hr + 1];
                const float P1 = zz[1][2 * hr] + zz[1][2 * hr + 1];
                float s0 = P0, s1 = P1;
                float y;
                y = __shfl_down_sync(kFull, s0, 1, 4); if (q < 3) s0 += y;
                y = __shfl_down_sync(kFull, s0, 2, 4); if (q < 2) s0 += y;
                y = __shfl_down_sync(kFull, s1, 1, 4); if (q < 3) s1 += y;
                y = __shfl_down_sync(kFull, s1, 2, 4); if (q < 2) s1 += y;
                const float upper = __shfl_sync(kFull, s1, 0, 4);
                const float lowAfter = s0 - P0, upAfter = s1 - P1;
                const float S9 = zz[1][2 * hr + 1] + upAfter + carry;
                const float S8 = zz[1][2 * hr] + S9;
                const float S1 = zz[0][2 * hr + 1] + lowAfter + upper + carry;
                const float S0v = zz[0][2 * hr] + S1;
                const float Sv[4] = {S0v, S1, S8, S9};
                const int tv[4] = {2 * q, 2 * q + 1, 8 + 2 * q, 9 + 2 * q};
                const float ev[4] = {ee[0][2 * hr], ee[0][2 * hr + 1], ee[1][2 * hr], ee[1][2 * hr + 1]};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = tv[m];
                    if (t < nv) {
                        const float d = dd[t * SP + row];
                        const float dp = t ? dd[(t - 1) * SP + row] : 1.f;
                        p.dw[base0 + (size_t)(t0 + t) * tstride + row] = (Sv[m] - ev[m]) * (dp * rcp_approx(d));
                    }
                }
                const float total = __shfl_sync(kFull, S0v, 0, 4);
                if (hr) carryB = total; else carryA = total;
            }
        }
        __syncthreads();  // raw no longer read
        if (c > 0) stage<E, 6, NT>(raw, src, base0 + (size_t)(t0 - C) * tstride, tstride, C);
        cp_async_commit();

        // G5: G_prev = G diag(d_C) + [DY | DSA] [R^ | A^]^T  (rows = value index)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float2 dc = *reinterpret_cast<const float2 *>(dC + 8 * nt + 2 * q);
            Gh[nt][0] *= dc.x; Gh[nt][1] *= dc.y; Gh[nt][2] *= dc.x; Gh[nt][3] *= dc.y;
            mma3(Gh[nt], dyA, ld_b(B5, (0 * 8 + nt) * 32 + lane));
            mma3(Gh[nt], dsA, ld_b(B5, (1 * 8 + nt) * 32 + lane));
        }
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

template <typename E>
cudaError_t launch_t(const SeqArgs &p, cudaStream_t st) {
    const size_t sm = bwd_smem_bytes<E>();
    cudaError_t e = cudaFuncSetAttribute(wkv7_bwd_chunk_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    wkv7_bwd_chunk_kernel<E><<<p.B * p.H, NT, sm, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool backward_chunk_supported(const SeqArgs &p) { return p.L == C; }

cudaError_t launch_backward_chunk(const SeqArgs &p, cudaStream_t st) {
    return p.dtype == 1 ? launch_t<__nv_bfloat16>(p, st) : launch_t<float>(p, st);
}

}  // namespace wkv7
