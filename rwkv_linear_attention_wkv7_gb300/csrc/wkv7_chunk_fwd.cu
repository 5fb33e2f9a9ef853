// Chunked WKV7 forward on warp-level tensor cores.
//
// Per (b,h) the recurrence S_t = S_{t-1} diag(w_t) + (S_{t-1} a_t) b_t^T
// + v_t k_t^T, y_t = S_t r_t (layouts of the "Foundry/cuda_kernels/timemix.cu"
// page) is evaluated 16 tokens at a time.  With the chunk notation of
// wkv7_chunk_common.cuh the chunk's sa_t solve a unit triangular 16x16 system
// and every state-dependent quantity is a dense contraction with the
// chunk-start state S_0:
//     SA  = S_0 A' + V M_k' = U W        U = S_0 A^ + V M_k,  W = (I - M_b)^{-1}
//     Y   = S_0 R' + V Q'   = Z + SA Q_b  Z = S_0 R^ + V Q_k
//     S_C = S_0 diag(d_C) + SA Bbar^T + V Kbar^T      (Bbar = B~ diag(d_C), Kbar = K~ diag(d_C))
// (A' = A^ W, M_k' = M_k W, R' = R^ + A' Q_b, Q' = Q_k + M_k' Q_b) and, since
// the column scaling commutes, S_C = (S_0 + SA B~^T + V K~^T) diag(d_C).  The
// large products U and Z need only the Gram, so they run while one warp
// solves for W; SA and Y then take two 16 x 16 products.  Every matrix
// operand is split into bf16 hi + lo once, into row-major shared matrices
// that ldmatrix (.trans where the use is transposed) turns into MMA
// fragments.  The state
// products run on mma.sync bf16 with split operands (three products) and
// fp32 accumulation; the state lives in registers as MMA accumulators: warp w
// owns value rows 16w..16w+15.  One CTA of 4 warps per (b,h), sized (registers
// and shared memory) so that four CTAs share an SM.
//
// A chunk whose cumulative decay leaves [1e-20, 1e20] (e.g. w = 0) cannot use
// 1/d_t; it takes the exact per-token recurrence on the same register layout.
//
// kGN: the output epilogue of the "timemix.cu" page (k_groupnorm, then
// k_bonus) is fused in: while a chunk's rows are staged, the bonus
// (sum_j r_j k_j r_k[j]) v of each token goes into a [C][64] tile; once the
// chunk's y is staged, the warps normalise each token over the head's 64
// outputs (biased variance, eps 64e-5, per-channel weight and bias; eight
// lanes per token) and adds the bonus in place; y and the epilogue output o
// leave by two tensor stores.
#include <type_traits>

#include "wkv7_chunk_common.cuh"

namespace wkv7 {
namespace {
using namespace chunk;

constexpr int NT = 128;
constexpr int YS = 68;  // row stride (floats) of the y staging block
// Lane 0 of warp 3 issues the y (and o) stores: warp 0 forms the inverse, the
// chunk's critical path.
constexpr int kYStoreThread = 96;
// Row pitch (floats) of the checkpoint staging: a half-warp's float2 stores of
// accumulator rows g, g + 1, ... then fall in distinct banks (with OS = 68 two
// rows four banks apart overlap).  Two warps' eight-row halves fill one split
// operand slot exactly.
constexpr int CKS = 72;

// Shared-memory carve-up (byte offsets after the raw input block).  HL16 = a
// split operand matrix (bf16 hi then lo) of 16 rows, row stride MS; HLC = a
// compact 16 x 16 split matrix, row stride CS.
constexpr int HL16 = 2 * 16 * MS * 2;
constexpr int HLC = 2 * 16 * CS * 2;
constexpr int B_DD = 0;                              // d fp32 [C][DS]
constexpr int B_BT = B_DD + C * SP * 4;              // b~ [t][j]
constexpr int B_KT = B_BT + HL16;                    // k~ [t][j]
constexpr int B_AH = B_KT + HL16;                    // a^ [t][j]
constexpr int B_RH = B_AH + HL16;                    // r^ [t][j]
constexpr int B_VM = B_RH + HL16;                    // v [t][i]
constexpr int B_Y = B_VM + HL16;                     // y staging fp32 [C][YS]
constexpr int B_QB = B_Y + C * YS * 4;               // Q_b [s][t]  (compact; Q_b, M_k, Q_k in
constexpr int B_MK = B_QB + HLC;                     // M_k [s][t]   the order of the Gram
constexpr int B_QK = B_MK + HLC;                     // Q_k [s][t]   warps 1, 2, 3)
constexpr int B_WT = B_QK + HLC;                     // W^T [t][s]  (compact)
constexpr int B_MB = B_WT + HLC;                     // M_b fp32 [C][MBS] (for the inverse)
constexpr int kBytes = B_MB + C * MBS * 4;
static_assert(2 * 8 * 72 * 4 <= HL16, "two warps' checkpoint halves fit one split operand slot");
static_assert(B_BT % 16 == 0 && B_Y % 128 == 0 && B_QB % 16 == 0 && B_MB % 16 == 0 && YS == OS,
              "aligned blocks; the y staging block is a tensor-store source");

constexpr int kBonusBytes = C * 64 * 4;  // kGN: bonus, then epilogue output, tile [C][64] fp32 (after kBytes)
template <typename E, bool kGN>
__host__ __device__ constexpr size_t fwd_smem_bytes() { return raw_bytes<E>() + (size_t)kBytes + (kGN ? kBonusBytes : 0); }

__device__ __forceinline__ HL hl(const unsigned char *base, int off) {
    const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(base + off);
    return HL{p, p + 16 * MS};
}
__device__ __forceinline__ HL hlc(const unsigned char *base, int off) {
    const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(base + off);
    return HL{p, p + 16 * CS};
}
__device__ __forceinline__ __nv_bfloat16 *hi_of(unsigned char *base, int off) {
    return reinterpret_cast<__nv_bfloat16 *>(base + off);
}
__device__ __forceinline__ __nv_bfloat16 *lo_of(unsigned char *base, int off) {
    return reinterpret_cast<__nv_bfloat16 *>(base + off) + 16 * MS;
}

// kP: the staged w, a, b rows hold the producers' inputs (w_pre, kk, avec); see in_w.
// kGN: the GroupNorm + bonus output epilogue (see the file header).
// kMode (for the time split's segment passes, which need only a segment's end
// state): 0 the whole forward; 1 the end state only (no y: r is not staged, and
// Z, Y, Q_b, Q_k are not formed); 2 the end state with v = 0, i.e. the product
// of the transitions applied to s0 (k and v are not staged either, M_k and
// every V product are skipped).
template <typename E, bool kP, bool kGN, int kMode = 0>
__global__ void __launch_bounds__(NT, 4) wkv7_fwd_chunk_kernel(SeqArgs p, const __grid_constant__ InputMaps maps) {
    static_assert(kMode == 0 || (!kP && !kGN), "the state-only passes run on plain inputs");
    extern __shared__ __align__(128) unsigned char smem[];
    // bf16 inputs: v is exact in bf16, so products with v as the A operand skip its (zero) lo part
    constexpr bool kVLo = !std::is_same<E, __nv_bfloat16>::value;
    E *raw = reinterpret_cast<E *>(smem);
    unsigned char *Bs = smem + raw_bytes<E>();
    float *dd = reinterpret_cast<float *>(Bs + B_DD), *ys = reinterpret_cast<float *>(Bs + B_Y);
    float *Mb = reinterpret_cast<float *>(Bs + B_MB);
    float *bon = reinterpret_cast<float *>(Bs + kBytes);  // kGN: bonus / epilogue output tile [C][64]
    const HL BT = hl(Bs, B_BT), KT = hl(Bs, B_KT), AH = hl(Bs, B_AH), RH = hl(Bs, B_RH), VM = hl(Bs, B_VM);
    const HL QB = hlc(Bs, B_QB), MK = hlc(Bs, B_MK), QK = hlc(Bs, B_QK), WT = hlc(Bs, B_WT);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int bh = blockIdx.x, bi = bh / p.H, h = bh % p.H;
    const size_t sbase = (size_t)bh * 64 * 64;
    const int rA = warp * 16 + g, rB = rA + 8;  // the two state rows this lane holds

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

    const int nchunks = (p.T + C - 1) / C;
    // chunk inputs arrive by tensor copies (one per input) on the TMA engine;
    // phase c of the mbarrier is chunk c
    __shared__ __align__(8) uint64_t bar;
    __shared__ int lost;  // a bounded wait of this CTA ran out (see mbar_wait)
    // the staged rows this mode reads: all six; w, k, v, a, b; or w, a, b
    constexpr unsigned kRows = kMode == 0 ? 6 : kMode == 1 ? 5 : 3;
    constexpr unsigned kChunkBytes = (unsigned)raw_bytes<E>() / 6 * kRows;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_expect_tx(&bar, kChunkBytes);  // chunk 0's bytes, before any copy is issued
        lost = 0;
    }
    __syncthreads();
    int stuck = -1;  // the chunk whose wait ran out
    auto staged = [](int vec) { return kMode == 0 || (vec != VR && (kMode == 1 || (vec != VK && vec != VV))); };
    // chunk c's copies, input 2 (w - 1) + l from lane l < 2 of warp w >= 1: warp 0, which
    // forms the inverse right after the copies are issued, issues none.  Thread 0
    // announced the bytes (before a block barrier that precedes every issue) and
    // arrives once.
    const int cvec = warp >= 1 && lane < 2 ? 2 * (warp - 1) + lane : -1;
    auto prefetch = [&](int c) {
        if (cvec >= 0 && staged(cvec)) tma_rows(raw + cvec * C * RS, &maps.m[cvec], h, c * C, bi, &bar);
        if (tid == 0) mbar_arrive(&bar);
    };
    prefetch(0);
    // kGN: bonus tile of the staged chunk, bon[t][j] = (sum_i r_i k_i r_k[i]) v_j; thread
    // (t = e / 16, j = 4 (e % 16)) sums its four channels, the 16 lanes of a token finish it
    auto write_bonus = [&]() {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int e = tid + NT * m, t = e >> 4, j = (e & 15) * 4;
            const float4 rr = ld_raw4(raw, VR, t, j), kq = ld_raw4(raw, VK, t, j);
            const float4 rk = __ldg(reinterpret_cast<const float4 *>(p.r_k + h * 64 + j));
            float sb = rr.x * kq.x * rk.x + rr.y * kq.y * rk.y + rr.z * kq.z * rk.z + rr.w * kq.w * rk.w;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) sb += __shfl_xor_sync(0xffffffffu, sb, o);
            const float4 vv = ld_raw4(raw, VV, t, j);
            *reinterpret_cast<float4 *>(bon + t * 64 + j) = make_float4(sb * vv.x, sb * vv.y, sb * vv.z, sb * vv.w);
        }
    };

    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        mbar_wait(&bar, c & 1, p.err, &lost);
        // this warp's checkpoint stores have left the a^ / r^ slots (the splits write
        // there after the barrier below)
        if (lane == 0) bulk_wait_read();
        if (tid == 0 && c + 1 < nchunks) mbar_expect_tx(&bar, kChunkBytes + (c == 0 ? kPhantomTx : 0u));

        // checkpoint of the state before token t0; written once the previous
        // chunk's state update has long completed, not at the chunk start where
        // it would wait on those MMAs
        auto write_ckpt = [&]() {
            if (p.ckpt && t0 % p.L == 0) {
                float *dst = p.ckpt + ((size_t)bh * p.nck + t0 / p.L) * 64 * 64;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    *reinterpret_cast<float2 *>(dst + rA * 64 + 8 * nt + 2 * q) = make_float2(S[nt][0], S[nt][1]);
                    *reinterpret_cast<float2 *>(dst + rB * 64 + 8 * nt + 2 * q) = make_float2(S[nt][2], S[nt][3]);
                }
            }
        };

        float *const fc = p.fac ? p.fac + ((size_t)bh * nchunks + c) * fac::kWords : nullptr;
        // the cumulative decays on warps 1 and 2 (lane 0 of warp 3 has just issued the y store)
        const bool exact = __syncthreads_or(prep_decay<kP>(raw, dd, nv, 32));
        if (lost) {  // every thread has passed its wait (the barrier above): leave together
            stuck = c;
            break;
        }
        if (!exact) {
            // ---- split the decay-scaled vectors and v once: [t][j] quads
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int e = tid + NT * m, t = e >> 4, j = (e & 15) * 4;
                const float4 d = *reinterpret_cast<const float4 *>(dd + t * DS + j);
                const float4 dp = t ? *reinterpret_cast<const float4 *>(dd + (t - 1) * DS + j) : make_float4(1.f, 1.f, 1.f, 1.f);
                const float4 id = rcp4(d);
                st_hl4(hi_of(Bs, B_BT), lo_of(Bs, B_BT), t, j, mul4(in_b4<kP>(raw, t, j), id));
                if (kMode < 2) st_hl4(hi_of(Bs, B_KT), lo_of(Bs, B_KT), t, j, mul4(ld_raw4(raw, VK, t, j), id));
                st_hl4(hi_of(Bs, B_AH), lo_of(Bs, B_AH), t, j, mul4(in_a4<kP>(raw, t, j), dp));
                if (kMode == 0) st_hl4(hi_of(Bs, B_RH), lo_of(Bs, B_RH), t, j, mul4(ld_raw4(raw, VR, t, j), d));
                if (kVLo && kMode < 2) st_hl4(hi_of(Bs, B_VM), lo_of(Bs, B_VM), t, j, ld_raw4(raw, VV, t, j));
            }
            if constexpr (kGN) write_bonus();
            // bf16 v is its own hi part: its A fragment (A[i][t] = v[t][i]) comes straight
            // from the staged input, before the barrier that lets the next chunk's copies in
            AFrag vA;
            if (!kVLo && kMode < 2) {
                const __nv_bfloat16 *rv = reinterpret_cast<const __nv_bfloat16 *>(raw) + VV * C * RS;
                vA = lda_t_hi(HL{rv, rv}, 16 * warp, 0, lane);
            }
            __syncthreads();
            // raw is no longer read in this chunk: fetch the next one now
            if (c + 1 < nchunks) prefetch(c + 1);

            // Gram [B~; K~] [A^; R^]^T (warp -> m-tile b~ | k~, n-tile pair a^ | r^) and
            // [Z | U] = S_0 [R^ | A^] in one pass over j: both take the same r^ / a^ fragments
            float ya[4][4] = {};
            {
                const int mt = warp >> 1;
                const bool rn = warp & 1;
                float acc[2][4] = {};
#pragma unroll
                // the Gram blocks each mode needs: M_b (warp 0) always, M_k (warp 2) unless v = 0,
                // Q_b and Q_k (warps 1, 3) only with y
                const bool gram = kMode == 0 || warp == 0 || (kMode == 1 && warp == 2);
                for (int kk = 0; kk < 4; ++kk) {
                    BFrag bq[4];
                    if (kMode == 0) ldb2(RH, 0, 16 * kk, lane, bq[0], bq[1]);
                    ldb2(AH, 0, 16 * kk, lane, bq[2], bq[3]);
                    if (gram) {
                        const AFrag af = lda(mt ? KT : BT, 0, 16 * kk, lane);
                        const BFrag gq[2] = {rn ? bq[0] : bq[2], rn ? bq[1] : bq[3]};
                        mma3n<2>(acc, af, gq);
                    }
                    const AFrag sf = a_from_acc(S, kk);
                    if (kMode == 0)
                        mma3n<4>(ya, sf, bq);
                    else
                        mma3n<2>(ya + 2, sf, bq + 2);  // U only
                }
                if (warp == 0) {  // b~ . a^ = M_b (its unused lower part too), fp32 for the inverse
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = 8 * u + 2 * q;
                        *reinterpret_cast<float2 *>(Mb + g * MBS + col) = make_float2(acc[u][0], acc[u][1]);
                        *reinterpret_cast<float2 *>(Mb + (g + 8) * MBS + col) = make_float2(acc[u][2], acc[u][3]);
                    }
                } else if (gram) {  // b~ . r^ = Q_b, k~ . a^ = M_k, k~ . r^ = Q_k: masked to [s <= t] ([s < t] for
                                    // M_k) and split into their compact operand matrices
                    const int strict = warp == 2;
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (g + 8 * (e >> 1) + strict > 8 * u + 2 * q + (e & 1)) acc[u][e] = 0.f;
                    unsigned char *dst = Bs + B_QB + (warp - 1) * HLC;
                    st_acc16<CS>(hi_of(dst, 0), reinterpret_cast<__nv_bfloat16 *>(dst) + 16 * CS, 0, 0, acc, lane);
                }
            }
            __syncthreads();

            // W on warp 0 while every warp adds V [Q_k | M_k] to [Z | U] (warp 0 follows
            // with its own rows once W is done)
            prep_inverse_t(Mb, hi_of(Bs, B_WT), reinterpret_cast<__nv_bfloat16 *>(Bs + B_WT) + 16 * CS);
            if (kVLo && kMode < 2) vA = lda_t(VM, 16 * warp, 0, lane);
            if constexpr (kMode == 0) {
                BFrag bq[4];
                ldb2_t<CS>(QK, 0, 0, lane, bq[0], bq[1]);
                ldb2_t<CS>(MK, 0, 0, lane, bq[2], bq[3]);
                mma3n<4, kVLo>(ya, vA, bq);
            } else if constexpr (kMode == 1) {  // V M_k into U only
                BFrag bq[2];
                ldb2_t<CS>(MK, 0, 0, lane, bq[0], bq[1]);
                mma3n<2, kVLo>(ya + 2, vA, bq);
            }
            if (tid == kYStoreThread) bulk_wait_read();  // the previous y tile has left the staging block
            __syncthreads();  // W

            // Checkpoint of S_0 (before P2 updates S): each warp stages its 16 rows,
            // 8 at a time, in its quarter of the a^ / r^ slots (free once every warp's
            // U/Z is done) and writes them with 2-D tensor stores; the second half
            // waits for the first to have left the staging block.
            const bool ck = p.ckpt && t0 % p.L == 0;
            float *const ckst = reinterpret_cast<float *>(Bs + (warp < 2 ? B_AH : B_RH)) + (warp & 1) * 8 * CKS;
            const int ckrow = (bh * p.nck + t0 / p.L) * 64 + 16 * warp;
            auto stage_ck = [&](int half) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
                    *reinterpret_cast<float2 *>(ckst + g * CKS + 8 * nt + 2 * q) =
                        make_float2(S[nt][2 * half], S[nt][2 * half + 1]);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&maps.m[7], ckst, ckrow + 8 * half);
                    bulk_commit();
                }
            };
            if (ck) stage_ck(0);

            // ---- SA = U W and Y = Z + SA Q_b (16 x 16 per warp)
            float sa[2][4] = {};
            {
                const AFrag ua = make_a(make_float2(ya[2][0], ya[2][1]), make_float2(ya[2][2], ya[2][3]),
                                        make_float2(ya[3][0], ya[3][1]), make_float2(ya[3][2], ya[3][3]));
                BFrag bw[2];
                ldb2<CS>(WT, 0, 0, lane, bw[0], bw[1]);  // B[s][t] = W[s][t] = W^T[t][s]
                mma3n<2>(sa, ua, bw);
            }
            const AFrag saf = make_a(make_float2(sa[0][0], sa[0][1]), make_float2(sa[0][2], sa[0][3]),
                                     make_float2(sa[1][0], sa[1][1]), make_float2(sa[1][2], sa[1][3]));
            BFrag qbf[2];
            if constexpr (kMode == 0) {
                ldb2_t<CS>(QB, 0, 0, lane, qbf[0], qbf[1]);
                mma3n<2>(ya, saf, qbf);  // Y (tiles 0, 1 of ya)
            }
            if (kMode == 0 && fc) {  // factor cache for the backward
                st_acc2(fc + fac::kSA + 256 * warp, sa[0], sa[1], lane);
                if (warp == 1) {  // M_k' = M_k W and Q' = Q_k + M_k' Q_b
                    const AFrag am = lda<CS>(MK, 0, 0, lane);
                    BFrag bw[2];
                    ldb2<CS>(WT, 0, 0, lane, bw[0], bw[1]);
                    float cm[2][4] = {};
                    mma3n<2>(cm, am, bw);
                    const AFrag amp = make_a(make_float2(cm[0][0], cm[0][1]), make_float2(cm[0][2], cm[0][3]),
                                             make_float2(cm[1][0], cm[1][1]), make_float2(cm[1][2], cm[1][3]));
                    float cq[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int tc = 8 * nt + 2 * q;
                        const float2 x = ld_hl<CS>(QK.hi, QK.lo, g, tc), z = ld_hl<CS>(QK.hi, QK.lo, g + 8, tc);
                        cq[nt][0] = x.x; cq[nt][1] = x.y; cq[nt][2] = z.x; cq[nt][3] = z.y;
                    }
                    mma3n<2>(cq, amp, qbf);
                    st_afrag(fc + fac::kMkA, amp, lane);
                    st_bfrags_acc(fc + fac::kQB, cq, lane);
                } else if (warp == 3) {  // W (A operand of W B~) and W Q_b
                    const AFrag wa = lda_t<CS>(WT, 0, 0, lane);  // A[s][t] = W[s][t] = W^T[t][s]
                    float cb[2][4] = {};
                    mma3n<2>(cb, wa, qbf);
                    st_afrag(fc + fac::kWA, wa, lane);
                    st_bfrags_acc(fc + fac::kWQbB, cb, lane);
                }
            }
            if (ck) {
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                stage_ck(1);
            }
            // ---- S_C = (S_0 + SA B~^T + V K~^T) diag(d_C)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                BFrag bb0, bb1;
                ldb2_t(BT, 16 * pp, 0, lane, bb0, bb1);
                const BFrag bq[2] = {bb0, bb1};
                mma3n<2>(S + 2 * pp, saf, bq);
                if constexpr (kMode < 2) {
                    BFrag kb0, kb1;
                    ldb2_t(KT, 16 * pp, 0, lane, kb0, kb1);
                    const BFrag kq[2] = {kb0, kb1};
                    mma3n<2, kVLo>(S + 2 * pp, vA, kq);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * pp + u;
                    const float2 dc = *reinterpret_cast<const float2 *>(dd + (C - 1) * DS + 8 * nt + 2 * q);
                    S[nt][0] *= dc.x; S[nt][1] *= dc.y; S[nt][2] *= dc.x; S[nt][3] *= dc.y;
                }
            }
            // y of the chunk -> staging [t][row]
            if constexpr (kMode == 0) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int t = 8 * nt + 2 * q;
                    ys[t * YS + rA] = ya[nt][0];
                    ys[(t + 1) * YS + rA] = ya[nt][1];
                    ys[t * YS + rB] = ya[nt][2];
                    ys[(t + 1) * YS + rB] = ya[nt][3];
                }
            }
        } else {
            // exact per-token recurrence for a chunk whose decay leaves the factorisable range
            if constexpr (kGN) write_bonus();
            write_ckpt();
            if (tid == kYStoreThread) bulk_wait_read();  // the previous y tile has left the staging block
            __syncthreads();
            for (int t = 0; t < nv; ++t) {
                float sa0 = 0.f, sa1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int j = 8 * nt + 2 * q;
                    const float a0 = in_a<kP>(raw, t, j), a1 = in_a<kP>(raw, t, j + 1);
                    sa0 = __fmaf_rn(S[nt][0], a0, __fmaf_rn(S[nt][1], a1, sa0));
                    sa1 = __fmaf_rn(S[nt][2], a0, __fmaf_rn(S[nt][3], a1, sa1));
                }
                sa0 += __shfl_xor_sync(0xffffffffu, sa0, 1);
                sa0 += __shfl_xor_sync(0xffffffffu, sa0, 2);
                sa1 += __shfl_xor_sync(0xffffffffu, sa1, 1);
                sa1 += __shfl_xor_sync(0xffffffffu, sa1, 2);
                // v and k are not staged with kMode 2 (v = 0), r only with kMode 0 (y)
                const float v0 = kMode < 2 ? ld_raw(raw, VV, t, rA) : 0.f;
                const float v1 = kMode < 2 ? ld_raw(raw, VV, t, rB) : 0.f;
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 8 * nt + 2 * q + e;
                        const float wv = in_w<kP>(raw, t, j), bv = in_b<kP>(raw, t, j);
                        const float kv = kMode < 2 ? ld_raw(raw, VK, t, j) : 0.f;
                        S[nt][e] = __fmaf_rn(S[nt][e], wv, __fmaf_rn(sa0, bv, __fmul_rn(v0, kv)));
                        S[nt][2 + e] = __fmaf_rn(S[nt][2 + e], wv, __fmaf_rn(sa1, bv, __fmul_rn(v1, kv)));
                        if (kMode == 0) {
                            const float rv = ld_raw(raw, VR, t, j);
                            y0 = __fmaf_rn(S[nt][e], rv, y0);
                            y1 = __fmaf_rn(S[nt][2 + e], rv, y1);
                        }
                    }
                }
                if (kMode == 0) {
                    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
                    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
                    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
                    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
                    if (q == 0) {
                        ys[t * YS + rA] = y0;
                        ys[t * YS + rB] = y1;
                    }
                }
            }
            __syncthreads();
            if (c + 1 < nchunks) prefetch(c + 1);
        }
        fence_proxy_async();  // the staged y tile is read by a tensor store
        __syncthreads();
        if constexpr (kGN) {  // o = GroupNorm(y) + bonus in place over the bonus tile: eight lanes per token,
                              // channels 4l..4l+3 and 32+4l..32+4l+3 each (the eight lanes' 16-byte accesses
                              // cover 128 contiguous bytes; the statistics take one round of three
                              // shuffle levels)
            const int t = tid >> 3, j0 = (tid & 7) * 4;
            const float4 ya0 = *reinterpret_cast<const float4 *>(ys + t * YS + j0);
            const float4 ya1 = *reinterpret_cast<const float4 *>(ys + t * YS + j0 + 32);
            const float yv[8] = {ya0.x, ya0.y, ya0.z, ya0.w, ya1.x, ya1.y, ya1.z, ya1.w};
            // one round of sums about a shift m0 (the token's first channel), so that the
            // moments of y - m0 do not cancel: mean = m0 + E[z], var = E[z^2] - E[z]^2
            const float m0 = __shfl_sync(0xffffffffu, yv[0], lane & ~7);
            float z[8], sz = 0.f, szz = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                z[i] = yv[i] - m0;
                sz += z[i];
                szz += z[i] * z[i];
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                sz += __shfl_xor_sync(0xffffffffu, sz, o);
                szz += __shfl_xor_sync(0xffffffffu, szz, o);
            }
            const float ez = sz * (1.f / 64.f);
            float cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) cv[i] = z[i] - ez;
            const float rstd = rsqrtf(fmaxf(szz * (1.f / 64.f) - ez * ez, 0.f) + kGnEps);
            const float4 *gw4 = reinterpret_cast<const float4 *>(p.gn_w + h * 64 + j0);
            const float4 *gb4 = reinterpret_cast<const float4 *>(p.gn_b + h * 64 + j0);
            float4 *ob = reinterpret_cast<float4 *>(bon + t * 64 + j0);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // channels j0 + 32 hf .. + 3: float4 index 8 hf
                const float4 gw = __ldg(gw4 + 8 * hf), gb = __ldg(gb4 + 8 * hf), bv = ob[8 * hf];
                const float *c = cv + 4 * hf;
                ob[8 * hf] = make_float4(c[0] * rstd * gw.x + gb.x + bv.x, c[1] * rstd * gw.y + gb.y + bv.y,
                                     c[2] * rstd * gw.z + gb.z + bv.z, c[3] * rstd * gw.w + gb.w + bv.w);
            }
            fence_proxy_async();
            __syncthreads();
        }
        if (kMode == 0 && tid == kYStoreThread) {  // y (and o) of the chunk: one tensor store each (tokens past T
                                                   // are not written)
            tma_store_rows(&maps.m[6], ys, h, t0, bi);
            if constexpr (kGN) tma_store_rows(&maps.m[8], bon, h, t0, bi);
            bulk_commit();
        }
    }
    if (lane == 0) bulk_wait_all();
    if (stuck >= 0) mbar_drain(&bar, stuck & 1);
    if (p.sT) {
        float *dst = p.sT + sbase;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<float2 *>(dst + rA * 64 + 8 * nt + 2 * q) = make_float2(S[nt][0], S[nt][1]);
            *reinterpret_cast<float2 *>(dst + rB * 64 + 8 * nt + 2 * q) = make_float2(S[nt][2], S[nt][3]);
        }
    }
}

template <typename E, bool kP, bool kGN, int kMode = 0>
cudaError_t launch_t(const SeqArgs &p, cudaStream_t st) {
    const size_t sm = fwd_smem_bytes<E, kGN>();
    InputMaps maps;  // six inputs, y (box OS), the checkpoints, and o (box 64) with kGN
    cudaError_t e = encode_input_maps(&maps, p, nullptr);
    if (e == cudaSuccess && kMode == 0) e = encode_rows_map(&maps.m[6], p.y, 4, p.B, p.T, p.H, OS);
    if (e == cudaSuccess && p.ckpt) e = encode_ckpt_map(&maps.m[7], p.ckpt, (long long)p.B * p.H * p.nck * 64, 8, CKS);
    if (e == cudaSuccess && kGN) e = encode_rows_map(&maps.m[8], p.o, 4, p.B, p.T, p.H, 64);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(wkv7_fwd_chunk_kernel<E, kP, kGN, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
    wkv7_fwd_chunk_kernel<E, kP, kGN, kMode><<<p.B * p.H, NT, sm, st>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace

bool forward_chunk_supported(const SeqArgs &p) { return p.L % C == 0; }

cudaError_t launch_forward_chunk(const SeqArgs &p, cudaStream_t st) {
    if (p.state_only == 1)
        return p.dtype == 1 ? launch_t<__nv_bfloat16, false, false, 1>(p, st) : launch_t<float, false, false, 1>(p, st);
    if (p.state_only == 2)
        return p.dtype == 1 ? launch_t<__nv_bfloat16, false, false, 2>(p, st) : launch_t<float, false, false, 2>(p, st);
    if (p.gn_w) return p.dtype == 1 ? launch_t<__nv_bfloat16, false, true>(p, st) : launch_t<float, false, true>(p, st);
    if (p.prod) return p.dtype == 1 ? launch_t<__nv_bfloat16, true, false>(p, st) : launch_t<float, true, false>(p, st);
    return p.dtype == 1 ? launch_t<__nv_bfloat16, false, false>(p, st) : launch_t<float, false, false>(p, st);
}

}  // namespace wkv7
