// Chunked WKV7 forward on warp-level tensor cores.
//
// Per (b,h) the recurrence S_t = S_{t-1} diag(w_t) + (S_{t-1} a_t) b_t^T
// + v_t k_t^T, y_t = S_t r_t (layouts of the "Foundry/cuda_kernels/timemix.cu"
// page) is evaluated 16 tokens at a time.  With the chunk notation of
// wkv7_chunk_common.cuh the chunk's sa_t solve a unit triangular 16x16 system
// and every state-dependent quantity is a dense contraction with the
// chunk-start state S_0:
//     SA  = S_0 A' + V M_k'              (A' = A^ W,  M_k' = M_k W,  W = (I - M_b)^{-1})
//     Y   = S_0 R' + V Q'                (R' = R^ + A' Q_b,  Q' = Q_k + M_k' Q_b)
//     S_C = S_0 diag(d_C) + SA Bbar^T + V Kbar^T      (Bbar = B~ diag(d_C), Kbar = K~ diag(d_C))
// Everything that does not involve S_0 (the Gram, W, A', R', M_k', Q') is
// built once per chunk, on tensor cores where it is a contraction, and every
// matrix operand is split into bf16 hi + lo once, into a fragment-major
// shared buffer (one 128-bit load per mma operand fragment).  The state
// products run on mma.sync bf16 with split operands (three products) and
// fp32 accumulation; the state lives in registers as MMA accumulators: warp w
// owns value rows 16w..16w+15.  One CTA of 4 warps per (b,h), sized (registers
// and shared memory) so that four CTAs share an SM.
//
// A chunk whose cumulative decay leaves [1e-20, 1e20] (e.g. w = 0) cannot use
// 1/d_t; it takes the exact per-token recurrence on the same register layout.
#include "wkv7_chunk_common.cuh"

namespace wkv7 {
namespace {
using namespace chunk;

constexpr int NT = 128;
constexpr int QS = 36;  // row stride of QM: [s][0..15] = Q', [s][16..31] = M_k'

// float offsets after the raw input block
constexpr int O_DD = 0;                  // d [C][SP]
constexpr int O_G = O_DD + C * SP;       // Gram [32][GS]; y staging [C][SP]
constexpr int O_W = O_G + C * SP;        // W [C][WS]
constexpr int O_QM = O_W + C * WS;       // [C][QS]
constexpr int O_AP = O_QM + C * QS;      // A' (warp-local exchange) [C][SP]
constexpr int O_P1B = O_AP + C * SP;     // u32 [4 kt][4 nt][32 lanes][4]: B of S_0 [R' | A']
constexpr int O_VB = O_P1B + 2048;       // u32 [4 nt][32][4]: B of V [Q' | M_k']
constexpr int O_P2B = O_VB + 512;        // u32 [2 kt][8 nt][32][4]: B of [SA | V] [Bbar ; Kbar]^T
constexpr int O_VAF = O_P2B + 2048;      // u32 [4 warps][32][8]: A fragments of V (hi[4], lo[4])
constexpr int kFloats = O_VAF + 1024;
static_assert(32 * GS <= C * SP, "Gram must fit its slot");
static_assert(O_P1B % 4 == 0 && O_VB % 4 == 0 && O_P2B % 4 == 0 && O_VAF % 4 == 0, "16-byte fragment buffers");

template <typename E>
__host__ __device__ constexpr size_t fwd_smem_bytes() { return raw_bytes<E>() + (size_t)kFloats * sizeof(float); }

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

template <typename E>
__global__ void __launch_bounds__(NT, 4) wkv7_fwd_chunk_kernel(SeqArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);
    float *F = reinterpret_cast<float *>(smem + raw_bytes<E>());
    float *dd = F + O_DD, *G = F + O_G, *ys = F + O_G, *Wm = F + O_W, *QM = F + O_QM, *AP = F + O_AP;
    uint32_t *P1B = reinterpret_cast<uint32_t *>(F + O_P1B);
    uint32_t *VBF = reinterpret_cast<uint32_t *>(F + O_VB);
    uint32_t *P2B = reinterpret_cast<uint32_t *>(F + O_P2B);
    uint32_t *VAF = reinterpret_cast<uint32_t *>(F + O_VAF);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int bh = blockIdx.x, bi = bh / p.H, h = bh % p.H;
    const size_t tstride = (size_t)p.H * 64;
    const size_t base0 = ((size_t)bi * p.T * p.H + h) * 64;
    const size_t sbase = (size_t)bh * 64 * 64;
    const int rA = warp * 16 + g, rB = rA + 8;  // the two state rows this lane holds

    // decay-scaled chunk vectors, computed where they are consumed
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
    stage<E, 6, NT>(raw, src, base0, tstride, min(C, p.T));
    cp_async_commit();

    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        cp_async_wait_all();
        __syncthreads();

        if (p.ckpt && t0 % p.L == 0) {  // state before token t0
            float *dst = p.ckpt + ((size_t)bh * p.nck + t0 / p.L) * 64 * 64;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                *reinterpret_cast<float2 *>(dst + rA * 64 + 8 * nt + 2 * q) = make_float2(S[nt][0], S[nt][1]);
                *reinterpret_cast<float2 *>(dst + rB * 64 + 8 * nt + 2 * q) = make_float2(S[nt][2], S[nt][3]);
            }
        }

        const bool exact = __syncthreads_or(prep_decay(raw, dd, nv));
        if (!exact) {
            // ---- Gram [B~; K~] [A^; R^]^T: warp -> m-tile (b~ | k~), two n-tiles (a^ | r^)
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
                    G[row * GS + col] = acc[u][0];
                    G[row * GS + col + 1] = acc[u][1];
                    G[(row + 8) * GS + col] = acc[u][2];
                    G[(row + 8) * GS + col + 1] = acc[u][3];
                }
            }
            // ---- B fragments of [Bbar ; Kbar]^T (k = token, n = key column) and A fragments of V
            {
                const float *dC = dd + (C - 1) * SP;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int f = tid + NT * m;  // 512 fragments
                    const int kk = f >> 8, nt = (f >> 5) & 7, ln = f & 31;
                    const int gg = ln >> 2, qq = ln & 3, j = 8 * nt + gg;
                    const int vec = kk ? VK : VB;
                    const float sc = dC[j];
                    float x[4];
                    const int s4[4] = {2 * qq, 2 * qq + 1, 2 * qq + 8, 2 * qq + 9};
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] = ld_raw(raw, vec, s4[e], j) * (sc * rcp_approx(dd[s4[e] * SP + j]));
                    reinterpret_cast<uint4 *>(P2B)[f] = pack_b(x[0], x[1], x[2], x[3]);
                }
                // A fragments of V for the 4 row blocks (rows = value index, k = token)
                const int rb = tid >> 5, gg = lane >> 2, qq = lane & 3;
                const int ra = 16 * rb + gg, rbb = ra + 8;
                const AFrag va = make_a(make_float2(ld_raw(raw, VV, 2 * qq, ra), ld_raw(raw, VV, 2 * qq + 1, ra)),
                                        make_float2(ld_raw(raw, VV, 2 * qq, rbb), ld_raw(raw, VV, 2 * qq + 1, rbb)),
                                        make_float2(ld_raw(raw, VV, 2 * qq + 8, ra), ld_raw(raw, VV, 2 * qq + 9, ra)),
                                        make_float2(ld_raw(raw, VV, 2 * qq + 8, rbb), ld_raw(raw, VV, 2 * qq + 9, rbb)));
                uint4 *vd = reinterpret_cast<uint4 *>(VAF) + (rb * 32 + lane) * 2;
                vd[0] = make_uint4(va.hi[0], va.hi[1], va.hi[2], va.hi[3]);
                vd[1] = make_uint4(va.lo[0], va.lo[1], va.lo[2], va.lo[3]);
            }
            __syncthreads();
            prep_inverse(G, Wm);
            __syncthreads();

            // ---- A' = W^T-weighted A^ and R' = R^ + Q_b^T A' on tensor cores
            //      (M = token, N = key column: warp w owns key columns 16w..16w+15)
            {
                AFrag wt;  // A[t][s] = W[s][t]
                {
                    const Frag2 f0 = split2(Wm[(2 * q) * WS + g], Wm[(2 * q + 1) * WS + g]);
                    const Frag2 f1 = split2(Wm[(2 * q) * WS + g + 8], Wm[(2 * q + 1) * WS + g + 8]);
                    const Frag2 f2_ = split2(Wm[(2 * q + 8) * WS + g], Wm[(2 * q + 9) * WS + g]);
                    const Frag2 f3 = split2(Wm[(2 * q + 8) * WS + g + 8], Wm[(2 * q + 9) * WS + g + 8]);
                    wt.hi[0] = f0.hi; wt.lo[0] = f0.lo; wt.hi[1] = f1.hi; wt.lo[1] = f1.lo;
                    wt.hi[2] = f2_.hi; wt.lo[2] = f2_.lo; wt.hi[3] = f3.hi; wt.lo[3] = f3.lo;
                }
                auto qb = [&](int s, int t) { return s <= t ? G[s * GS + 16 + t] : 0.f; };  // Q_b[s][t]
                AFrag qbt;  // A[t][s] = Q_b[s][t]
                {
                    const Frag2 f0 = split2(qb(2 * q, g), qb(2 * q + 1, g));
                    const Frag2 f1 = split2(qb(2 * q, g + 8), qb(2 * q + 1, g + 8));
                    const Frag2 f2_ = split2(qb(2 * q + 8, g), qb(2 * q + 9, g));
                    const Frag2 f3 = split2(qb(2 * q + 8, g + 8), qb(2 * q + 9, g + 8));
                    qbt.hi[0] = f0.hi; qbt.lo[0] = f0.lo; qbt.hi[1] = f1.hi; qbt.lo[1] = f1.lo;
                    qbt.hi[2] = f2_.hi; qbt.lo[2] = f2_.lo; qbt.hi[3] = f3.hi; qbt.lo[3] = f3.lo;
                }
                float ca[2][4], cr[2][4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int jn = 16 * warp + 8 * u + g;  // B column (key) of this lane
                    ca[u][0] = ca[u][1] = ca[u][2] = ca[u][3] = 0.f;
                    mma3(ca[u], wt, make_b(make_float2(a_hat(2 * q, jn), a_hat(2 * q + 1, jn)),
                                           make_float2(a_hat(2 * q + 8, jn), a_hat(2 * q + 9, jn))));
                    const int jc = 16 * warp + 8 * u + 2 * q;  // C columns of this lane
                    *reinterpret_cast<float2 *>(AP + g * SP + jc) = make_float2(ca[u][0], ca[u][1]);
                    *reinterpret_cast<float2 *>(AP + (g + 8) * SP + jc) = make_float2(ca[u][2], ca[u][3]);
                }
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int jn = 16 * warp + 8 * u + g, jc = 16 * warp + 8 * u + 2 * q;
                    cr[u][0] = r_hat(g, jc); cr[u][1] = r_hat(g, jc + 1);
                    cr[u][2] = r_hat(g + 8, jc); cr[u][3] = r_hat(g + 8, jc + 1);
                    mma3(cr[u], qbt, make_b(make_float2(AP[(2 * q) * SP + jn], AP[(2 * q + 1) * SP + jn]),
                                            make_float2(AP[(2 * q + 8) * SP + jn], AP[(2 * q + 9) * SP + jn])));
                }
                // B fragments of S_0 [R' | A']: k-tile = warp, register half = u, n-tile = token half (+2 for A')
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const Frag2 r0 = split2(cr[u][0], cr[u][1]), r1 = split2(cr[u][2], cr[u][3]);
                    const Frag2 a0 = split2(ca[u][0], ca[u][1]), a1 = split2(ca[u][2], ca[u][3]);
                    uint32_t *base = P1B + (warp * 4) * 128 + lane * 4;
                    base[0 * 128 + u] = r0.hi; base[0 * 128 + 2 + u] = r0.lo;
                    base[1 * 128 + u] = r1.hi; base[1 * 128 + 2 + u] = r1.lo;
                    base[2 * 128 + u] = a0.hi; base[2 * 128 + 2 + u] = a0.lo;
                    base[3 * 128 + u] = a1.hi; base[3 * 128 + 2 + u] = a1.lo;
                }
            }
            if (warp == 0) {  // M_k' = M_k W and Q' = Q_k + M_k' Q_b (16 x 16), then the V-side B fragments
                auto mk = [&](int s, int u) { return u > s ? G[(16 + s) * GS + u] : 0.f; };  // M_k[s][u]
                const AFrag am = make_a(make_float2(mk(g, 2 * q), mk(g, 2 * q + 1)), make_float2(mk(g + 8, 2 * q), mk(g + 8, 2 * q + 1)),
                                        make_float2(mk(g, 2 * q + 8), mk(g, 2 * q + 9)),
                                        make_float2(mk(g + 8, 2 * q + 8), mk(g + 8, 2 * q + 9)));
                float cm[2][4] = {};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int t = 8 * nt + g;
                    mma3(cm[nt], am, make_b(make_float2(Wm[(2 * q) * WS + t], Wm[(2 * q + 1) * WS + t]),
                                            make_float2(Wm[(2 * q + 8) * WS + t], Wm[(2 * q + 9) * WS + t])));
                }
                const AFrag amp = make_a(make_float2(cm[0][0], cm[0][1]), make_float2(cm[0][2], cm[0][3]),
                                         make_float2(cm[1][0], cm[1][1]), make_float2(cm[1][2], cm[1][3]));
                auto qbv = [&](int u, int t) { return u <= t ? G[u * GS + 16 + t] : 0.f; };       // Q_b[u][t]
                auto qkv = [&](int s, int t) { return s <= t ? G[(16 + s) * GS + 16 + t] : 0.f; };  // Q_k[s][t]
                float cq[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int tc = 8 * nt + 2 * q, t = 8 * nt + g;
                    cq[nt][0] = qkv(g, tc); cq[nt][1] = qkv(g, tc + 1); cq[nt][2] = qkv(g + 8, tc); cq[nt][3] = qkv(g + 8, tc + 1);
                    mma3(cq[nt], amp, make_b(make_float2(qbv(2 * q, t), qbv(2 * q + 1, t)),
                                             make_float2(qbv(2 * q + 8, t), qbv(2 * q + 9, t))));
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int tc = 8 * nt + 2 * q;
                    QM[g * QS + tc] = cq[nt][0]; QM[g * QS + tc + 1] = cq[nt][1];
                    QM[(g + 8) * QS + tc] = cq[nt][2]; QM[(g + 8) * QS + tc + 1] = cq[nt][3];
                    QM[g * QS + 16 + tc] = cm[nt][0]; QM[g * QS + 16 + tc + 1] = cm[nt][1];
                    QM[(g + 8) * QS + 16 + tc] = cm[nt][2]; QM[(g + 8) * QS + 16 + tc + 1] = cm[nt][3];
                }
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int n = 8 * nt + g;
                    reinterpret_cast<uint4 *>(VBF)[nt * 32 + lane] =
                        pack_b(QM[(2 * q) * QS + n], QM[(2 * q + 1) * QS + n], QM[(2 * q + 8) * QS + n], QM[(2 * q + 9) * QS + n]);
                }
            }
            __syncthreads();
            // raw is no longer read in this chunk: fetch the next one under the state products
            if (c + 1 < nchunks) stage<E, 6, NT>(raw, src, base0 + (size_t)(t0 + C) * tstride, tstride, min(C, p.T - t0 - C));
            cp_async_commit();

            // ---- [Y | SA] = S_0 [R' | A'] + V [Q' | M_k']
            float ya[4][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const AFrag sf = a_from_acc(S, kk);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) mma3(ya[nt], sf, ld_b(P1B, (kk * 4 + nt) * 32 + lane));
            }
            AFrag vA;
            {
                const uint4 *vs = reinterpret_cast<const uint4 *>(VAF) + (warp * 32 + lane) * 2;
                const uint4 h4 = vs[0], l4 = vs[1];
                vA.hi[0] = h4.x; vA.hi[1] = h4.y; vA.hi[2] = h4.z; vA.hi[3] = h4.w;
                vA.lo[0] = l4.x; vA.lo[1] = l4.y; vA.lo[2] = l4.z; vA.lo[3] = l4.w;
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma3(ya[nt], vA, ld_b(VBF, nt * 32 + lane));

            // ---- S_C = S_0 diag(d_C) + [SA | V] [Bbar^T ; Kbar^T]
            const AFrag saf = make_a(make_float2(ya[2][0], ya[2][1]), make_float2(ya[2][2], ya[2][3]),
                                     make_float2(ya[3][0], ya[3][1]), make_float2(ya[3][2], ya[3][3]));
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const float2 dc = *reinterpret_cast<const float2 *>(dd + (C - 1) * SP + 8 * nt + 2 * q);
                S[nt][0] *= dc.x; S[nt][1] *= dc.y; S[nt][2] *= dc.x; S[nt][3] *= dc.y;
                mma3(S[nt], saf, ld_b(P2B, (0 * 8 + nt) * 32 + lane));
                mma3(S[nt], vA, ld_b(P2B, (1 * 8 + nt) * 32 + lane));
            }
            // y of the chunk -> staging [t][row] (the Gram slot is free now)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t = 8 * nt + 2 * q;
                ys[t * SP + rA] = ya[nt][0];
                ys[(t + 1) * SP + rA] = ya[nt][1];
                ys[t * SP + rB] = ya[nt][2];
                ys[(t + 1) * SP + rB] = ya[nt][3];
            }
        } else {
            // exact per-token recurrence for a chunk whose decay leaves the factorisable range
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
            if (c + 1 < nchunks) stage<E, 6, NT>(raw, src, base0 + (size_t)(t0 + C) * tstride, tstride, min(C, p.T - t0 - C));
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

template <typename E>
cudaError_t launch_t(const SeqArgs &p, cudaStream_t st) {
    const size_t sm = fwd_smem_bytes<E>();
    cudaError_t e = cudaFuncSetAttribute(wkv7_fwd_chunk_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    wkv7_fwd_chunk_kernel<E><<<p.B * p.H, NT, sm, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool forward_chunk_supported(const SeqArgs &p) { return p.L % C == 0; }

cudaError_t launch_forward_chunk(const SeqArgs &p, cudaStream_t st) {
    return p.dtype == 1 ? launch_t<__nv_bfloat16>(p, st) : launch_t<float>(p, st);
}

}  // namespace wkv7
