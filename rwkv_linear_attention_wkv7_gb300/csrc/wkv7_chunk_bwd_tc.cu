// Chunked WKV7 backward with the 64-row state products that feed only the
// gradient outputs on the fifth-generation tensor cores (tcgen05.mma,
// accumulators in tensor memory).
//
// The algebra is that of wkv7_chunk_bwd.cu (the adjoint of the recurrence, the
// "WKV kernel backward" block of accumulate_token_step_gradients on the
// "infotheory/backends/rwkvzip/rwkv7/model.rs" page, evaluated one 16-token
// chunk at a time in reverse from the forward's stride-16 checkpoints and its
// per-chunk factor cache).  Of the contractions over a whole 64-row state,
// the two that carry the state gradient from chunk to chunk,
//   G2  [DV | DSA] = G [K' | B'] + ...     G5  G_prev = G d_C + [DY | DSA] [R^ | A^]^T,
// stay on warp-level mma.sync spread over the four warps: as chains of
// single-thread tcgen05.mma (12 and 6 dependent MMAs of about 50 cycles each)
// they lengthened every chunk's critical path and the kernel measured slower
// (3.53 ms on the bf16 B=16 T=4096 H=32 workload, against 2.67 ms for the
// warp-level kernel as it then was).  The two that only feed the gradient
// outputs,
//   G3  S_0^T [DY | DSA]   (M = 64 keys, N = 32, K = 64 value rows)
//   G4  G^T [V | SA]       (M = 64 keys, N = 32, K = 64 value rows; scaled by d_C per key after)
// are issued by one thread as tcgen05.mma (bf16 operands split hi + lo, three
// products per K step, fp32 accumulation in TMEM) as soon as their operands
// exist, from matrices the warps write into shared memory in the canonical
// core-matrix layout of wkv7_tc.cuh, and run while the warps do G2, Gam, G5 and
// the masked products; the warps read them back at the gradient epilogue with
// tcgen05.ld in the accumulator-fragment layout of mma.sync.  Needs the
// forward's factor cache (stride 16).
#include <type_traits>

#include "wkv7_chunk_bwd_exact.cuh"
#include "wkv7_tc.cuh"

namespace wkv7 {
namespace {
using namespace chunk;

// Shared-memory carve-up (byte offsets after the raw input block).  Split
// operand matrices are canonical (hi part, then lo part).
constexpr int HL64C = 2 * 64 * 64 * 2;          // 64 x 64 split matrix
constexpr int HL32C = 2 * 32 * 64 * 2;          // 32 x 64 split matrix
constexpr int HLM = 2 * 32 * 32 * 2;            // 32 x 32 split matrix (masked Gam blocks)
constexpr int B_DYF = 0;                        // dy fp32 [C][SP] (tensor copy)
constexpr int B_DD = B_DYF + C * SP * 4;        // d fp32 [C][DS]
constexpr int B_CAR = B_DD + C * SP * 4;        // dw carry partials of the last chunk, 4 x 64 fp32
constexpr int B_FAC = B_CAR + 1024;             // factor block of the chunk (bulk copy)
constexpr int B_S0 = B_FAC + fac::kWords * 4;   // S_0 split [i][j]; then the dr, dw, dk staging tiles
constexpr int B_GS = B_S0 + HL64C;              // G split [i][j]; exact path: S_{t-1} (over GS and BK)
constexpr int B_BK = B_GS + HL64C;              // [B~; K~] rows t (b~ 0..15, k~ 16..31), columns j
constexpr int B_RA = B_BK + HL32C;              // [R^; A^]; exact path: column partial sums
constexpr int B_VS = B_RA + HL32C;              // [V; SA] rows t, columns i; then the dv staging tile
constexpr int B_DY = B_VS + HL32C;              // [DY; DSA]; then the da staging tile
constexpr int B_KB = B_DY + HL32C;              // [K'; B']; then M3 | M4; then the db staging tile
constexpr int kBytes = B_KB + HL32C;
constexpr int kTile = 1152;                     // floats between staging tiles ([C][OS] fp32 each)
static_assert(B_S0 % 1024 == 0 && B_GS % 1024 == 0 && B_VS % 1024 == 0 && B_DY % 1024 == 0 && B_KB % 1024 == 0,
              "operand matrices and staging tiles aligned");
static_assert(3 * kTile * 4 <= HL64C && C * OS * 4 <= kTile * 4 && C * OS * 4 <= HL32C, "staging tiles fit");
static_assert(64 * SP * 4 <= HL64C + HL32C && 5 * 4 * 64 * 4 <= HL32C, "exact-path scratch fits");
static_assert(2 * HLM <= HL32C, "M3 and M4 fit the [K'; B'] slot");

// TMEM columns of the accumulators
constexpr int kColG3 = 0, kColG4 = 32, kColST = 64, kCols = 128;
constexpr uint32_t kIdN32MK = tc::idesc_bf16(64, 32, 1, 0);  // G3, G4: A MN-major, B K-major
constexpr uint32_t kIdN64MM = tc::idesc_bf16(64, 64, 1, 1);  // sT: A and B MN-major

template <typename E>
__host__ __device__ constexpr size_t bwd_tc_smem_bytes() { return raw_bytes<E>() + (size_t)kBytes; }

__device__ __forceinline__ HL hlc(const unsigned char *base, int off, int elems) {
    const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(base + off);
    return HL{p, p + elems};
}
__device__ __forceinline__ __nv_bfloat16 *mut(const __nv_bfloat16 *p) { return const_cast<__nv_bfloat16 *>(p); }
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// kP: the staged w, a, b rows hold the producers' inputs (w_pre, kk, avec; see
// in_w) and dw, da, db receive dw_pre, dkk, davec; sigmoid(w_pre) terms and
// avec at each lane's epilogue positions are kept in registers from the split
// phase, since the staged rows are refilled before the epilogue.
template <typename E, bool kP>
__global__ void __launch_bounds__(NT, 2)
    wkv7_bwd_tc_kernel(SeqArgs p, const __grid_constant__ InputMaps maps, const __grid_constant__ OutputMaps omaps) {
    constexpr bool kVLo = !std::is_same<E, __nv_bfloat16>::value;  // bf16 v: its lo part is zero
    extern __shared__ __align__(1024) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);
    unsigned char *Bs = smem + raw_bytes<E>();
    float *dyf = reinterpret_cast<float *>(Bs + B_DYF), *dd = reinterpret_cast<float *>(Bs + B_DD);
    float *car = reinterpret_cast<float *>(Bs + B_CAR);
    const float *FC = reinterpret_cast<const float *>(Bs + B_FAC);
    const HL S0H = hlc(Bs, B_S0, 64 * 64), GS = hlc(Bs, B_GS, 64 * 64), BK = hlc(Bs, B_BK, 32 * 64),
             RA = hlc(Bs, B_RA, 32 * 64), VS = hlc(Bs, B_VS, 32 * 64), DY = hlc(Bs, B_DY, 32 * 64),
             KB = hlc(Bs, B_KB, 32 * 64), M3 = hlc(Bs, B_KB, 32 * 32), M4 = hlc(Bs, B_KB + HLM, 32 * 32);

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

    const int nchunks = (p.T + C - 1) / C;
    // bar: a chunk's inputs, dy and factor block (phase k = the chunk processed k-th);
    // g3, g4: the tensor-core products (phase = the tensor-core chunks done so far);
    // x: the last chunk's sT product; dr: the final drain before TMEM is released
    __shared__ __align__(8) uint64_t bar, bar_g3, bar_g4, bar_x, bar_dr;
    __shared__ uint32_t tmem_slot;
    __shared__ int lost;  // a bounded wait of this CTA ran out (see mbar_wait)
    if (warp == 0) tc::alloc(&tmem_slot, kCols);
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init(&bar_g3, 1);
        mbar_init(&bar_g4, 1);
        mbar_init(&bar_x, 1);
        mbar_init(&bar_dr, 1);
        lost = 0;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tb = tmem_slot;
    int stuck = -1, mph = 0;

    constexpr unsigned kChunkBytes = (unsigned)(raw_bytes<E>() + C * RS * 4 + fac::kWords * 4);
    auto stage_in = [&](int c) {  // inputs and dy of chunk c (lanes 0..6 of warp 0), factor block (lane 3)
        if (tid < 7) {
            void *const dst = tid < 6 ? static_cast<void *>(raw + tid * C * RS) : static_cast<void *>(dyf);
            tma_rows(dst, &maps.m[tid], h, c * C, bi, &bar);
        }
        if (tid == 3) bulk_g2s(Bs + B_FAC, p.fac_in + ((size_t)bh * nchunks + c) * fac::kWords, fac::kWords * 4, &bar);
        if (tid == 0) mbar_arrive(&bar);
    };
    const float *ck0 = p.ckpt_in + (size_t)bh * p.nck * 4096;  // this head's checkpoints
    if (tid == 0) mbar_expect_tx(&bar, kChunkBytes);
    stage_in(nchunks - 1);
    if (tid == 0) bulk_prefetch_l2(ck0 + (size_t)(nchunks - 1) * 4096, 4096 * 4);

    // shared-memory addresses of the operand parts, for the MMA descriptors
    const uint32_t aS0h = tc::saddr(S0H.hi), aS0l = tc::saddr(S0H.lo), aGh = tc::saddr(GS.hi), aGl = tc::saddr(GS.lo);
    const uint32_t aBKh = tc::saddr(BK.hi), aBKl = tc::saddr(BK.lo), aRAh = tc::saddr(RA.hi), aRAl = tc::saddr(RA.lo);
    const uint32_t aVSh = tc::saddr(VS.hi), aVSl = tc::saddr(VS.lo), aDYh = tc::saddr(DY.hi), aDYl = tc::saddr(DY.lo);
    const bool store_lane = (warp == 0 && lane < 4) || (warp == 1 && lane < 2);

    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        const bool last = c == nchunks - 1;
        const unsigned ph = (nchunks - 1 - c) & 1;
        mbar_wait(&bar, ph, p.err, &lost);
        if (tid == 0 && c > 0) mbar_expect_tx(&bar, kChunkBytes + (last ? kPhantomTx : 0u));
        // the chunk-start state from its checkpoint (L2, prefetched a chunk ago): lane
        // segment s = rows (s & 7) + 8 (s >> 6), columns 8 ((s >> 3) & 7) .. + 7
        float4 s0v[8];
        {
            const float *src = ck0 + (size_t)c * 4096;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s = tid + NT * k, i = (s & 7) + 8 * (s >> 6), cg = (s >> 3) & 7;
                s0v[2 * k] = __ldg(reinterpret_cast<const float4 *>(src + i * 64 + 8 * cg));
                s0v[2 * k + 1] = __ldg(reinterpret_cast<const float4 *>(src + i * 64 + 8 * cg + 4));
            }
        }
        if (tid == 0 && c > 0) bulk_prefetch_l2(ck0 + (size_t)(c - 1) * 4096, 4096 * 4);
        // the previous chunk's gradient stores have read the staging tiles the splits refill
        if (store_lane) bulk_wait_read();
        // the cumulative decays on warps 2 and 3
        const bool exact = __syncthreads_or(prep_decay<kP, E, !kP>(raw, dd, nv, 64));
        if (lost) {  // every thread has passed its wait (the barrier above): leave together
            stuck = c;
            break;
        }
        if (exact) {
            bwd_chunk_exact<E, kP, 64>(raw, dyf, ck0 + (size_t)c * 4096, reinterpret_cast<float *>(Bs + B_GS),
                                       reinterpret_cast<float *>(Bs + B_RA), Gh, nv, p, base0, tstride, t0, carryA,
                                       carryB);
            fence_proxy_async();  // the per-token path wrote into slots the copies refill
            __syncthreads();
            if (c > 0) stage_in(c - 1);
            continue;
        }
        const float *dC = dd + (C - 1) * DS;

        // ================= operand matrices (split once, canonical layout)
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // b~, k~, r^, a^ of this warp's 16-key slab, all tokens: a quarter-warp
                                       // takes 8 tokens of one quad, a half-warp both quads of one core
                                       // matrix, so that every access falls in distinct banks
            const int t = (lane & 7) + 8 * m, j = 16 * warp + 4 * ((lane >> 3) & 1) + 8 * (lane >> 4);
            const float4 d = *reinterpret_cast<const float4 *>(dd + t * DS + j);
            const float4 dp = t ? *reinterpret_cast<const float4 *>(dd + (t - 1) * DS + j) : make_float4(1.f, 1.f, 1.f, 1.f);
            const float4 id = rcp4(d);
            tc::st_hl4<64>(mut(BK.hi), mut(BK.lo), t, j, mul4(in_b4<kP>(raw, t, j), id));
            tc::st_hl4<64>(mut(BK.hi), mut(BK.lo), 16 + t, j, mul4(ld_raw4(raw, VK, t, j), id));
            tc::st_hl4<64>(mut(RA.hi), mut(RA.lo), t, j, mul4(ld_raw4(raw, VR, t, j), d));
            tc::st_hl4<64>(mut(RA.hi), mut(RA.lo), 16 + t, j, mul4(in_a4<kP>(raw, t, j), dp));
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // dy and v rows: lanes cover two core matrices (256 contiguous bytes)
            const int e = tid + NT * m;
            const int t = ((e >> 1) & 7) + 8 * (e >> 7), i = 8 * ((e >> 4) & 7) + 4 * (e & 1);
            tc::st_hl4<64>(mut(DY.hi), mut(DY.lo), t, i, *reinterpret_cast<const float4 *>(dyf + t * SP + i));
            tc::st_hl4<64>(mut(VS.hi), mut(VS.lo), t, i, ld_raw4(raw, VV, t, i));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // S_0
            const int s = tid + NT * k, i = (s & 7) + 8 * (s >> 6), cg = (s >> 3) & 7;
            tc::st_hl8<64>(mut(S0H.hi), mut(S0H.lo), i, 8 * cg, s0v[2 * k], s0v[2 * k + 1]);
        }
#pragma unroll
        for (int pp = 0; pp < 4; ++pp)  // G (this warp's 16 value rows)
            tc::st_acc16<64>(mut(GS.hi), mut(GS.lo), 16 * warp, 16 * pp, Gh + 2 * pp, lane);
        float sa[2][4];  // SA from the forward -> [V; SA] rows 16..31 (transposed)
        ld_acc2(FC + fac::kSA + 256 * warp, sa[0], sa[1], lane);
        tc::st_acc_t16<64>(mut(VS.hi), mut(VS.lo), 16, 16 * warp, sa, lane);
        // kP: -0.606531 sigmoid (1 - sigmoid) of w_pre at this lane's dw positions (keys rA / rB,
        // tokens 2q, 2q + 1, 8 + 2q, 9 + 2q) and avec at its da positions (tokens 8nt + 2q + (m & 1),
        // keys rA for m < 2, rB otherwise), taken while the staged rows are this chunk's
        float sgf[2][4], avf[2][4];
        if constexpr (kP) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = 8 * (m >> 1) + 2 * q + (m & 1);
                    const float sg = sigmoid_f(ld_raw(raw, VW, t, hr ? rB : rA));
                    sgf[hr][m] = -kDecayScale * sg * (1.f - sg);
                }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int m = 0; m < 4; ++m) avf[nt][m] = ld_raw(raw, VB, 8 * nt + 2 * q + (m & 1), m < 2 ? rA : rB);
        }
        __syncwarp();  // this warp's b~ / k~ slab is all its K' / B' products read
        {   // K' = d_C o (K~ + M_k' B~), B' = d_C o (W B~) (M = token, N = key; warp w owns keys 16w..)
            const AFrag amk = ld_afrag(FC + fac::kMkA, lane), awn = ld_afrag(FC + fac::kWA, lane);
            BFrag b0, b1;
            tc::ldb2_t<64>(BK, 16 * warp, 0, lane, b0, b1);
            float ck[2][4], cb2[2][4] = {};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int jc = 16 * warp + 8 * u + 2 * q;
                const float2 k0 = tc::ld_hl<64>(BK, 16 + g, jc), k8 = tc::ld_hl<64>(BK, 24 + g, jc);
                ck[u][0] = k0.x; ck[u][1] = k0.y; ck[u][2] = k8.x; ck[u][3] = k8.y;
            }
            const BFrag bq[2] = {b0, b1};
            mma3n<2>(ck, amk, bq);
            mma3n<2>(cb2, awn, bq);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float2 dc = *reinterpret_cast<const float2 *>(dC + 16 * warp + 8 * u + 2 * q);
                ck[u][0] *= dc.x; ck[u][1] *= dc.y; ck[u][2] *= dc.x; ck[u][3] *= dc.y;
                cb2[u][0] *= dc.x; cb2[u][1] *= dc.y; cb2[u][2] *= dc.x; cb2[u][3] *= dc.y;
            }
            tc::st_acc16<64>(mut(KB.hi), mut(KB.lo), 0, 16 * warp, ck, lane);    // K' rows (tokens)
            tc::st_acc16<64>(mut(KB.hi), mut(KB.lo), 16, 16 * warp, cb2, lane);  // B' rows
        }
        // every operand of G4 (and sT) is written: hand them to the tensor cores
        fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // G4: D[j][t'] = sum_i G[i][j] [V; SA][t'][i]
                tc::mma3(tb + kColG4, tc::mndesc<64>(aGh, ks), tc::mndesc<64>(aGl, ks), tc::kdesc<64>(aVSh, ks),
                         tc::kdesc<64>(aVSl, ks), kIdN32MK, ks > 0);
            tc::commit(&bar_g4);
            if (last && p.dsT) {  // sT - S_0 = V K~^T + SA B~^T before the d_C scaling: D[i][j]
                tc::mma3(tb + kColST, tc::mndesc<64>(aVSh, 0), tc::mndesc<64>(aVSl, 0), tc::mndesc<64>(aBKh, 1),
                         tc::mndesc<64>(aBKl, 1), kIdN64MM, false);
                tc::mma3(tb + kColST, tc::mndesc<64>(aVSh, 1), tc::mndesc<64>(aVSl, 1), tc::mndesc<64>(aBKh, 0),
                         tc::mndesc<64>(aBKl, 0), kIdN64MM, true);
                tc::commit(&bar_x);
            }
        }

        // ================= G2: [DV | DSA] = G [K' | B'] + DY [Q'^T | (W Q_b)^T] (value rows)
        float dvs[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag gf = a_from_acc(Gh, kk);
            BFrag b0, b1, b2, b3;
            tc::ldb2<64>(KB, 0, 16 * kk, lane, b0, b1);
            tc::ldb2<64>(KB, 16, 16 * kk, lane, b2, b3);
            const BFrag bq[4] = {b0, b1, b2, b3};
            mma3n<4>(dvs, gf, bq);
        }
        const AFrag dyA = tc::lda_t<64>(DY, 16 * warp, 0, lane);  // A[i][t] = DY[t][i]
        {
            BFrag b0, b1, b2, b3;
            ld_bfrags(FC + fac::kQB, lane, b0, b1);
            ld_bfrags(FC + fac::kWQbB, lane, b2, b3);
            const BFrag bq[4] = {b0, b1, b2, b3};
            mma3n<4>(dvs, dyA, bq);
        }
        // the dw running sum starts at diag(dsT^T sT): sT = (S_0 + V K~^T + SA B~^T) diag(d_C)
        if (last && p.dsT) {
            mbar_wait(&bar_x, 0, p.err, &lost);
            tc::fence_after();
            const float *s0g = ck0 + (size_t)c * 4096;
            float part[8][2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[4][4];
                tc::ld32(tc::taddr(tb, warp, kColST + 32 * half), x);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int nt = 4 * half + u, j0 = 8 * nt + 2 * q;
                    const float2 sA = __ldg(reinterpret_cast<const float2 *>(s0g + rA * 64 + j0));
                    const float2 sB = __ldg(reinterpret_cast<const float2 *>(s0g + rB * 64 + j0));
                    const float2 dc = *reinterpret_cast<const float2 *>(dC + j0);
                    const float ST[4] = {(sA.x + x[u][0]) * dc.x, (sA.y + x[u][1]) * dc.y, (sB.x + x[u][2]) * dc.x,
                                         (sB.y + x[u][3]) * dc.y};
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        part[nt][e] = rows_sum(__fmaf_rn(Gh[nt][e], ST[e], __fmul_rn(Gh[nt][2 + e], ST[2 + e])));
                }
            }
            if (g == 0) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    car[warp * 64 + 8 * nt + 2 * q] = part[nt][0];
                    car[warp * 64 + 8 * nt + 2 * q + 1] = part[nt][1];
                }
            }
            __syncthreads();
            carryA = car[rA] + car[64 + rA] + car[128 + rA] + car[192 + rA];
            carryB = car[rB] + car[64 + rB] + car[128 + rB] + car[192 + rB];
        }
        // DSA -> [DY; DSA] rows 16..31 (DSA[i][t] -> row 16 + t, column i)
        tc::st_acc_t16<64>(mut(DY.hi), mut(DY.lo), 16, 16 * warp, dvs + 2, lane);
        const AFrag dsA = make_a(make_float2(dvs[2][0], dvs[2][1]), make_float2(dvs[2][2], dvs[2][3]),
                                 make_float2(dvs[3][0], dvs[3][1]), make_float2(dvs[3][2], dvs[3][3]));
        fence_proxy_async();
        tc::fence_before();
        __syncthreads();  // DSA visible; every warp is past its [K'; B'] reads
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // G3: D[j][t'] = sum_i S_0[i][j] [DY; DSA][t'][i]
                tc::mma3(tb + kColG3, tc::mndesc<64>(aS0h, ks), tc::mndesc<64>(aS0l, ks), tc::kdesc<64>(aDYh, ks),
                         tc::kdesc<64>(aDYl, ks), kIdN32MK, ks > 0);
            tc::commit(&bar_g3);
        }
        if (c > 0) stage_in(c - 1);  // the staged rows, dy and factors of this chunk are consumed

        {   // Gam = [SA | V]^T [DY | DSA] (32 x 32): warp -> m-tile (SA | V), n-tile pair (DY | DSA),
            // written into its two masked split blocks (the [K'; B'] slot: every warp is past G2)
            //   M3[k][n] = Gam[k][n] where (n < 16 ? s <= t : s < t)           (s = k % 16, t = n % 16)
            //   M4[k][n] = Gam[n < 16 ? 16 + t : t][k] where (k < 16 ? s >= t : s > t)
            const int mt = warp >> 1;
            float acc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                BFrag bq[4];
                tc::ldb2<64>(DY, 0, 16 * kk, lane, bq[0], bq[1]);
                tc::ldb2<64>(DY, 16, 16 * kk, lane, bq[2], bq[3]);
                const AFrag af = (mt && !kVLo) ? tc::lda_hi<64>(VS, 0, 16 * kk, lane)
                                               : tc::lda<64>(VS, mt ? 0 : 16, 16 * kk, lane);
                const bool ds = warp & 1;
                const BFrag gq[2] = {ds ? bq[2] : bq[0], ds ? bq[3] : bq[1]};
                mma3n<2>(acc, af, gq);
            }
            float m3[2][4], m4[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int R = 16 * mt + g + 8 * hr;              // Gam row
                    const int Cc = 16 * (warp & 1) + 8 * u + 2 * q;  // Gam column (even)
                    const int s3 = R & 15;
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int n = Cc + z, t = n & 15;
                        const float x = acc[u][2 * hr + z];
                        m3[u][2 * hr + z] = (n >= 16 ? s3 < t : s3 <= t) ? x : 0.f;
                        m4[u][2 * hr + z] = ((n >= 16) ? (t > s3) : (t >= s3)) ? x : 0.f;
                    }
                }
            tc::st_acc16<32>(mut(M3.hi), mut(M3.lo), 16 * mt, 16 * (warp & 1), m3, lane);
            tc::st_acc_t16<32>(mut(M4.hi), mut(M4.lo), 16 * (warp & 1), mt ? 0 : 16, m4, lane);
        }
        // ================= G5: G_prev = G d_C + [DY | DSA] [R^ | A^]^T (value rows)
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            BFrag rr[2], aa[2];
            tc::ldb2_t<64>(RA, 16 * pp, 0, lane, rr[0], rr[1]);
            tc::ldb2_t<64>(RA, 16 * pp, 16, lane, aa[0], aa[1]);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int nt = 2 * pp + u;
                const float2 dc = *reinterpret_cast<const float2 *>(dC + 8 * nt + 2 * q);
                Gh[nt][0] *= dc.x; Gh[nt][1] *= dc.y; Gh[nt][2] *= dc.x; Gh[nt][3] *= dc.y;
            }
            mma3n<2>(Gh + 2 * pp, dyA, rr);
            mma3n<2>(Gh + 2 * pp, dsA, aa);
        }
        __syncthreads();  // masked Gam blocks visible

        // ================= [DR | DA] (key rows): [B~ | K~] M3 + S_0^T [DY | DSA]
        const AFrag btA = tc::lda_t<64>(BK, 16 * warp, 0, lane), ktA = tc::lda_t<64>(BK, 16 * warp, 16, lane);
        float x3[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            BFrag bq[4];
            tc::ldb2_t<32>(M3, 0, 16 * kk, lane, bq[0], bq[1]);
            tc::ldb2_t<32>(M3, 16, 16 * kk, lane, bq[2], bq[3]);
            mma3n<4>(x3, kk ? ktA : btA, bq);
        }
        // ================= [DK | DB] (key rows): [R^ | A^] M4 + d_C o (G^T [V | SA])
        const AFrag rhA = tc::lda_t<64>(RA, 16 * warp, 0, lane), ahA = tc::lda_t<64>(RA, 16 * warp, 16, lane);
        float x4[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            BFrag bq[4];
            tc::ldb2_t<32>(M4, 0, 16 * kk, lane, bq[0], bq[1]);
            tc::ldb2_t<32>(M4, 16, 16 * kk, lane, bq[2], bq[3]);
            mma3n<4>(x4, kk ? ahA : rhA, bq);
        }
        mbar_wait(&bar_g3, mph & 1, p.err, &lost);
        mbar_wait(&bar_g4, mph & 1, p.err, &lost);
        tc::fence_after();
        {
            float t3[4][4], t4[4][4];
            tc::ld32(tc::taddr(tb, warp, kColG3), t3);
            tc::ld32(tc::taddr(tb, warp, kColG4), t4);
            const float dcA = dC[rA], dcB = dC[rB];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                x3[n][0] += t3[n][0]; x3[n][1] += t3[n][1]; x3[n][2] += t3[n][2]; x3[n][3] += t3[n][3];
                x4[n][0] = __fmaf_rn(dcA, t4[n][0], x4[n][0]);
                x4[n][1] = __fmaf_rn(dcA, t4[n][1], x4[n][1]);
                x4[n][2] = __fmaf_rn(dcB, t4[n][2], x4[n][2]);
                x4[n][3] = __fmaf_rn(dcB, t4[n][3], x4[n][3]);
            }
        }
        ++mph;

        // ================= gradients: staged as [t][key] tiles (stride OS) in slots whose
        // readers are done (S_0: G3; [V; SA]: G4 and Gam; [DY; DSA]: G3, G5 and Gam; M3 | M4),
        // then one tensor store each
        __syncthreads();  // every warp is past its M3 / M4 reads
        float *const gdr = reinterpret_cast<float *>(Bs + B_S0), *const gdw = gdr + kTile, *const gdk = gdr + 2 * kTile;
        float *const gdv = reinterpret_cast<float *>(Bs + B_VS), *const gda = reinterpret_cast<float *>(Bs + B_DY);
        float *const gdb = reinterpret_cast<float *>(Bs + B_KB);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {  // dv (rows of G2 = value index)
            const int t = 8 * nt + 2 * q;
            gdv[t * OS + rA] = dvs[nt][0];
            gdv[(t + 1) * OS + rA] = dvs[nt][1];
            gdv[t * OS + rB] = dvs[nt][2];
            gdv[(t + 1) * OS + rB] = dvs[nt][3];
        }
        {
            // r^, a^, b~, k~ at this lane's (token, key) positions, in accumulator order
            float rv[8], av[8], bv[8], kv[8];
            a_values(rhA, rv);
            a_values(ahA, av);
            a_values(btA, bv);
            a_values(ktA, kv);
            float zz[2][4], ee[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int vi = 4 * nt + m;  // value index in a_values order
                    const int row = m < 2 ? rA : rB;
                    const int t = 8 * nt + 2 * q + (m & 1);
                    const float d = dd[t * DS + row];
                    const float dp = t ? dd[(t - 1) * DS + row] : 1.f;
                    const float inv = rcp_approx(d);
                    const float xr = x3[nt][m], xa = x3[nt + 2][m], xk = x4[nt][m], xb = x4[nt + 2][m];
                    // r o dr = r^ o X3_r, a o da = a^ o X3_a, b o db = b~ o X4_b, k o dk = k~ o X4_k
                    ee[nt][m] = av[vi] * xa;
                    zz[nt][m] = rv[vi] * xr + ee[nt][m] - bv[vi] * xb - kv[vi] * xk;
                    gdr[t * OS + row] = d * xr;
                    gdk[t * OS + row] = inv * xk;
                    if constexpr (kP) {  // dkk = -da + avec db, davec = kk db (k_comp_keymod)
                        const float db_ = inv * xb;
                        gda[t * OS + row] = avf[nt][m] * db_ - dp * xa;
                        gdb[t * OS + row] = -av[vi] * rcp_approx(dp) * db_;
                    } else {
                        gda[t * OS + row] = dp * xa;
                        gdb[t * OS + row] = inv * xb;
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
                    const float d = dd[t * DS + row];
                    const float dp = t ? dd[(t - 1) * DS + row] : 1.f;
                    if constexpr (kP) {  // dw_pre = (w o dw) (-0.606531) sigmoid (1 - sigmoid) (k_wdecay_bwd)
                        gdw[t * OS + row] = (Sv[m] - ev[m]) * sgf[hr][m];
                    } else {
                        gdw[t * OS + row] = (Sv[m] - ev[m]) * (dp * rcp_approx(d));
                    }
                }
                const float total = __shfl_sync(kFull, S0v, 0, 4);
                if (hr) carryB = total; else carryA = total;
            }
        }

        fence_proxy_async();  // the staged tiles are read by the tensor stores
        __syncthreads();
        // one tensor store per lane: dr, dw, dk, dv from lanes 0..3 of warp 0, da, db
        // from lanes 0..1 of warp 1
        if (store_lane) {
            const int o = warp == 0 ? lane : 4 + lane;
            const float *const tile = o < 3 ? gdr + kTile * o : o == 3 ? gdv : o == 4 ? gda : gdb;
            tma_store_rows(&omaps.m[o], tile, h, t0, bi);
            bulk_commit();
        }
    }
    if (store_lane) bulk_wait_all();
    if (stuck >= 0) mbar_drain(&bar, (nchunks - 1 - stuck) & 1);
    if (tid == 0) {  // no MMA may still run when its tensor memory is released
        tc::commit(&bar_dr);
        mbar_drain(&bar_dr, 0);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::dealloc(tb, kCols);
    if (p.ds0) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<float2 *>(p.ds0 + sbase + rA * 64 + 8 * nt + 2 * q) = make_float2(Gh[nt][0], Gh[nt][1]);
            *reinterpret_cast<float2 *>(p.ds0 + sbase + rB * 64 + 8 * nt + 2 * q) = make_float2(Gh[nt][2], Gh[nt][3]);
        }
    }
}

template <typename E, bool kP>
cudaError_t launch_t(const SeqArgs &p, cudaStream_t st) {
    const size_t sm = bwd_tc_smem_bytes<E>();
    InputMaps maps;
    OutputMaps omaps;
    cudaError_t e = encode_input_maps(&maps, p, p.dy);  // six inputs and dy
    if (e == cudaSuccess) e = encode_output_maps(&omaps, p);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(wkv7_bwd_tc_kernel<E, kP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    wkv7_bwd_tc_kernel<E, kP><<<p.B * p.H, NT, sm, st>>>(p, maps, omaps);
    return cudaGetLastError();
}

}  // namespace

bool backward_tc_supported(const SeqArgs &p) { return p.L == C && p.fac_in != nullptr; }

cudaError_t launch_backward_tc(const SeqArgs &p, cudaStream_t st) {
    if (p.prod) return p.dtype == 1 ? launch_t<__nv_bfloat16, true>(p, st) : launch_t<float, true>(p, st);
    return p.dtype == 1 ? launch_t<__nv_bfloat16, false>(p, st) : launch_t<float, false>(p, st);
}

}  // namespace wkv7
