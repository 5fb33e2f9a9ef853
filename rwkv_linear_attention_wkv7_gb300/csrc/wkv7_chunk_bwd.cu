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
// ([DV | DSA] is evaluated as X = Gd [K~ | B~]^T, DV = X_K + X_B M_k'^T + DY Q'^T,
// DSA = X_B W^T + DY Q_b'^T: K' and B' are never formed.)
// dw needs no contraction of its own: summing H_t o S_t over the value rows
// in two ways gives, per key column,
//   w_t o dw_t = r_t o dr_t - b_t o db_t - k_t o dk_t + (w o dw + a o da)_{t+1},
// a reverse running sum whose value past the last token is diag(dsT^T sT).
// Chunks whose decay underflows take an exact per-token path that replays
// the chunk from its checkpoint.
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "wkv7_chunk_bwd_exact.cuh"

// The state-gradient instantiation (kSO) ends each chunk after its chain, so
// the later phases of the chunk loop are unreachable there by design.
#pragma nv_diag_suppress 128

namespace wkv7 {
namespace {
using namespace chunk;

// Shared-memory carve-up (byte offsets after the raw input block).  HL16 /
// HL32 / HL64 = split operand matrices (bf16 hi then lo) of 16 / 32 / 64 rows
// with row stride MS.
constexpr int HL16 = 2 * 16 * MS * 2, HL32 = 2 * HL16, HL64 = 2 * HL32;
constexpr int B_DYF = 0;                       // dy fp32 [C][SP]        (chunk start .. conversion)
constexpr int B_DD = B_DYF + C * SP * 4;       // d fp32 [C][SP]
constexpr int B_G = B_DD + C * SP * 4;         // Gram, then Gam, fp32 [32][GS] (slot C*SP floats)
constexpr int B_W = B_G + C * SP * 4;          // W fp32 [C][WS]
constexpr int B_SX = B_W + 1280;               // S_0 fp32 [64][OS], then G d_C (HL64), then gradient staging
constexpr int B_BT = B_SX + HL64;              // b~, k~, a^, r^ (HL16 each) [t][j]; exact path: S_{t-1} fp32
constexpr int B_KT = B_BT + HL16;
constexpr int B_AH = B_KT + HL16;
constexpr int B_RH = B_AH + HL16;
constexpr int B_VV = B_RH + HL16;              // v [t][i]
constexpr int B_DYH = B_VV + HL16;             // dy [t][i]
constexpr int B_SAH = B_DYH + HL16;            // SA [t][i]
constexpr int B_DSH = B_SAH + HL16;            // DSA [t][i]
constexpr int B_Y = B_DSH + HL16;              // A' [t][j] (HL16), M_k' [s][t] (HL16), an HL32 slot, [Q'; W Q_b] (HL32)
constexpr int B_AP = B_Y, B_MK = B_Y + HL16, B_QQ = B_Y + 2 * HL32;
constexpr int B_M3 = B_Y, B_M4 = B_Y + HL32;   // masked Gam blocks [k][n] (HL32 each), after G1/G2
constexpr int kBytes = B_QQ + HL32;
static_assert(B_SX % 16 == 0 && B_BT % 16 == 0 && B_Y % 16 == 0, "16-byte aligned operand matrices");
static_assert(32 * GS <= C * SP && C * WS * 4 <= 1280, "small fp32 blocks fit");
static_assert(B_SX % 128 == 0 && B_VV % 128 == 0 && B_SAH % 128 == 0 && C * OS * 4 <= HL16,
              "gradient staging blocks: 128-byte aligned, one per 4.5 KiB slot");
static_assert(64 * OS * 4 <= HL64, "S_0 staging and the G d_C split share one slot");
static_assert(4 * HL16 >= 64 * SP * 4, "exact-path S_{t-1} fits the four scaled blocks");
static_assert(5 * 4 * 64 * 4 <= 2 * HL32, "exact-path scratch fits region Y");

// The state-gradient pass (kSO below) keeps only what its chain reads, contiguous: dy, the
// decays, the b~, a^, r^ and dy splits, and the first half of the factor block.
constexpr int S_BT = B_DD + C * SP * 4, S_AH = S_BT + HL16, S_RH = S_AH + HL16, S_DYH = S_RH + HL16,
              S_QQ = S_DYH + HL16;
constexpr int kStateBytes = S_QQ + fac::kSA * 4;
static_assert(B_G == S_BT && S_BT % 16 == 0 && S_QQ % 16 == 0, "state-pass layout: aligned, after dy and the decays");

// kGN: the head's gn_w and r_k (64 floats each) past the block, read by the do -> dy conversion
// at every chunk start (shared memory instead of a global load on the chunk's critical path)
constexpr int kGnParamBytes = 2 * 64 * 4;

template <typename E, bool kSO = false, bool kGN = false>
__host__ __device__ constexpr size_t bwd_smem_bytes() {
    return raw_bytes<E>() + (size_t)(kSO ? kStateBytes : kBytes) + (kGN ? kGnParamBytes : 0);
}

__device__ __forceinline__ HL hl(const unsigned char *base, int off, int rows) {
    const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(base + off);
    return HL{p, p + rows * MS};
}
__device__ __forceinline__ __nv_bfloat16 *hi_of(unsigned char *base, int off) {
    return reinterpret_cast<__nv_bfloat16 *>(base + off);
}
__device__ __forceinline__ __nv_bfloat16 *lo_of(unsigned char *base, int off, int rows) {
    return reinterpret_cast<__nv_bfloat16 *>(base + off) + rows * MS;
}
// An A fragment of a 16 x 16 matrix holds the B fragments of its transpose:
// n-tile n is registers n and n + 2.
__device__ __forceinline__ BFrag tb(const AFrag &a, int n) {
    BFrag b;
    b.hi[0] = a.hi[n]; b.hi[1] = a.hi[n + 2];
    b.lo[0] = a.lo[n]; b.lo[1] = a.lo[n + 2];
    return b;
}

// Token of element quad e (0..63) when a warp converts its own 16-key slab
// (4 quads per token): the 16 lanes of a half-warp take tokens 2 apart and
// the 8 of a quarter-warp tokens 4 apart, so that their 8-byte accesses to
// rows of 72 bf16 and their 16-byte accesses to rows of 68 floats fall in
// distinct banks.
__device__ __forceinline__ int slab_token(int e) {
    return 4 * ((e >> 2) & 1) + 2 * ((e >> 3) & 1) + ((e >> 4) & 1) + 8 * (e >> 5);
}

// A' = W^T-weighted a^ for NS 16-key slabs starting at slab0 (M = token,
// N = key), the slabs' MMAs issued together; written split to the A' slot.
template <int NS>
__device__ __forceinline__ void build_ap(const AFrag &wt, const HL &AH, unsigned char *Bs, int slab0, int lane) {
    const int g = lane >> 2, q = lane & 3;
    float ca[NS][2][4] = {};
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        BFrag b0, b1;
        ldb2_t(AH, 16 * (slab0 + s), 0, lane, b0, b1);
        mma3(ca[s][0], wt, b0);
        mma3(ca[s][1], wt, b1);
    }
    __nv_bfloat16 *ah = hi_of(Bs, B_AP), *al = lo_of(Bs, B_AP, 16);
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int jc = 16 * (slab0 + s) + 8 * u + 2 * q;
            st_hl(ah, al, g, jc, ca[s][u][0], ca[s][u][1]);
            st_hl(ah, al, g + 8, jc, ca[s][u][2], ca[s][u][3]);
        }
}

// kFac: the per-chunk factors (W, M_k', Q', W Q_b, SA) come from the
// forward's factor cache, prefetched into the [Q'; W Q_b] slot, instead of
// being rebuilt from the Gram (no Gram, inverse, A' or G1 in this mode).
// kP: the staged w, a, b rows hold the producers' inputs (w_pre, kk, avec; see
// in_w) and dw, da, db receive their gradients dw_pre, dkk, davec.  That
// epilogue runs after the staged rows are refilled: it takes kk from the a^
// split (a^ = -kk d_{t-1}), sigmoid(w_pre) (1 - sigmoid(w_pre)) from registers
// each lane fills from w_pre before the refill, and avec from a copy the split
// phase keeps in the Gram / W slots, which the factor-cache path does not use
// otherwise.
// kGN (with kFac, without kP): the backward of the GroupNorm + bonus output
// epilogue ("timemix.cu" page, k_bonus_bwd and k_groupnorm_bwd) is fused in
// front: the staged dy rows hold do = dL/do and the forward's y of the chunk
// arrives in the Gram slot (idle on the factor-cache path); 16 lanes per
// token turn do into the recurrence's dy in place (GroupNorm backward,
// reductions over the head's 64 channels), leave do s (the bonus's dv) in the
// y slot and sum_j do_j v_j per token for the bonus's dr and dk, and
// accumulate the parameter gradients of their four channels over every token;
// per-(b,h) partial sums leave at the end (summed over batch rows by
// wkv7_gn_param_reduce_kernel, no atomics).
// kSO (with kFac, without kP or kGN): the state gradient alone, ds0 (what a
// segment of a sequence sends to its start).  The adjoint does not depend on
// the state, so only the chain  DSA = X_B W^T + DY (W Q_b)^T,
// G_prev = Gd + [DY | DSA] [R^ | A^]^T  runs: no start state, no k or v, no SA,
// Gam or per-token gradient.  Its operations are those of the full kernel, in
// the same order, so ds0 is bit-identical to it.
template <typename E, bool kFac, bool kP, bool kGN, bool kSO = false>
__global__ void __launch_bounds__(NT, 2)
    wkv7_bwd_chunk_kernel(SeqArgs p, const __grid_constant__ InputMaps maps, const __grid_constant__ OutputMaps omaps) {
    static_assert(!kGN || (kFac && !kP), "the epilogue's backward runs on the factor-cache path without producers");
    static_assert(!kSO || (kFac && !kP && !kGN), "the state-gradient pass runs on the factor cache, plain inputs");
    // bf16 inputs: v is exact in bf16, so products with v as an operand skip its (zero) lo part
    constexpr bool kVLo = !std::is_same<E, __nv_bfloat16>::value;
    extern __shared__ __align__(128) unsigned char smem[];
    E *raw = reinterpret_cast<E *>(smem);
    unsigned char *Bs = smem + raw_bytes<E>();
    float *dyf = reinterpret_cast<float *>(Bs + B_DYF), *dd = reinterpret_cast<float *>(Bs + B_DD);
    float *Gm = reinterpret_cast<float *>(Bs + B_G), *Wm = reinterpret_cast<float *>(Bs + B_W);
    // kP: avec of the chunk, fp32 [C][OS], past the 256 floats the last chunk's dw carry uses
    float *const avs = Gm + 256;
    // kP: sigmoid(w_pre) of the chunk, fp32 [C][DS], from the decay phase to the dw_pre
    // factors (the slot takes the masked Gam block M4 only after those are formed)
    float *const sgs = reinterpret_cast<float *>(Bs + B_M4);
    static_assert(C * DS * 4 <= HL32, "the sigmoid block fits the M4 slot");
    static_assert(256 * 4 + C * OS * 4 <= C * SP * 4 + 1280, "avec copy fits the Gram and W slots");
    float *S0f = reinterpret_cast<float *>(Bs + B_SX);
    constexpr int oBT = kSO ? S_BT : B_BT, oAH = kSO ? S_AH : B_AH, oRH = kSO ? S_RH : B_RH;
    constexpr int oDYH = kSO ? S_DYH : B_DYH, oQQ = kSO ? S_QQ : B_QQ;
    const HL SX = hl(Bs, B_SX, 64), BT = hl(Bs, oBT, 16), KT = hl(Bs, B_KT, 16), AH = hl(Bs, oAH, 16),
             RH = hl(Bs, oRH, 16), VM = hl(Bs, B_VV, 16), DYH = hl(Bs, oDYH, 16), SAH = hl(Bs, B_SAH, 16),
             DSH = hl(Bs, B_DSH, 16), AP = hl(Bs, B_AP, 16), MK = hl(Bs, B_MK, 16),
             QQ = hl(Bs, B_QQ, 32), M3 = hl(Bs, B_M3, 32), M4 = hl(Bs, B_M4, 32);

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
    // A chunk's inputs and dy (tensor copies) and factor block (bulk copy)
    // arrive on the TMA engine, completed on one mbarrier whose phase k holds
    // the chunk processed k-th (nchunks - 1 - c).  Thread 0 announces the bytes
    // right after the previous phase completed and arrives once the inputs are
    // issued.  The chunk's start state comes on a second mbarrier (same phase
    // numbering): one 2-D tensor copy of the fp32 checkpoint into the S_0 slot
    // (rows of stride OS, the columns past 64 zero fill), issued at the chunk
    // start once the previous chunk's gradient stores have read their staging
    // there, and first waited for by the products that read S_0.
    __shared__ __align__(8) uint64_t bar, bar_s;
    __shared__ int lost;  // a bounded wait of this CTA ran out (see mbar_wait)
    // kSO stages neither k nor v, and of the factor block only its first half (W, M_k', Q', W Q_b)
    constexpr int kFacWords = kSO ? fac::kSA : fac::kWords;
    constexpr unsigned kChunkBytes = (unsigned)(raw_bytes<E>() - (kSO ? 2 * C * RS * sizeof(E) : 0) + C * RS * 4 +
                                                (kFac ? kFacWords * 4 : 0) + (kGN ? C * RS * 4 : 0));
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init(&bar_s, 1);
        mbar_expect_tx(&bar, kChunkBytes);  // the last chunk's bytes, before any copy is issued
        lost = 0;
    }
    __syncthreads();
    int stuck = -1, s_phase = -1;  // the chunk whose wait ran out; the phase of the last start-state copy
    // kGN: parameter-gradient sums of this lane's channels 4 (lane % 16) .. + 3 (over the
    // tokens it converts), the bonus weights of its key rows rA, rB; per-token
    // sum_j do_j v_j past the dw carry in the W slot
    float4 pgw = {}, pgb = {}, prk = {};
    float rkA = 0.f, rkB = 0.f;
    float *const dsv = Wm + 256;
    static_assert(256 * 4 + C * 4 <= 1280, "the dw carry and the per-token sums fit the W slot");
    float *const gnp = reinterpret_cast<float *>(Bs + kBytes);  // kGN: gn_w [64], r_k [64]
    if constexpr (kGN) {
        if (tid < 32) {
            const float *src = tid < 16 ? p.gn_w + h * 64 + 4 * tid : p.r_k + h * 64 + 4 * (tid - 16);
            *reinterpret_cast<float4 *>(gnp + 4 * tid) = __ldg(reinterpret_cast<const float4 *>(src));
        }
        rkA = __ldg(p.r_k + h * 64 + rA);
        rkB = __ldg(p.r_k + h * 64 + rB);
    }
    // the last chunk's dw carry partials: the Gram slot, or the W slot when the Gram slot stages y
    float *const carp = kGN ? Wm : Gm;
    constexpr unsigned kS0Bytes = 64 * OS * 4;
    // A chunk's copies come from lanes 0..2 of warps 1..3, copy 3 (w - 1) + l: the six
    // inputs, dy, the factor block, and (kGN) the forward's y.  Warp 0 issues the
    // gradient stores and the start-state copy; thread 0 announces the bytes (before a
    // block barrier that precedes every issue) and arrives once.
    const int ccopy = warp >= 1 && lane < 3 ? 3 * (warp - 1) + lane : -1;
    auto stage_in = [&](int c) {  // inputs and dy of chunk c (and y): one tensor copy each
        if (ccopy >= 0 && ccopy < 7 && !(kSO && (ccopy == VK || ccopy == VV))) {
            void *const dst = ccopy < 6 ? static_cast<void *>(raw + ccopy * C * RS) : static_cast<void *>(dyf);
            tma_rows(dst, &maps.m[ccopy], h, c * C, bi, &bar);
        }
        if constexpr (kGN) {
            if (ccopy == 8) tma_rows(Gm, &maps.m[8], h, c * C, bi, &bar);
        }
    };
    auto load_s0 = [&](int c) {  // thread 0
        s_phase = (nchunks - 1 - c) & 1;
        mbar_expect_tx(&bar_s, kS0Bytes);
        tma_load_2d(S0f, &maps.m[7], (bh * p.nck + c) * 64, &bar_s);
        mbar_arrive(&bar_s);
    };
    // S_0 operand fragments straight from the fp32 staging, split on the way:
    // A[m][k] = S_0[m0 + m][k0 + k] (s0_a) or S_0[k0 + k][m0 + m] (s0_at).
    // Rows of stride OS put the 32 lanes' words in distinct banks.
    auto ld2 = [](const float *x) { return *reinterpret_cast<const float2 *>(x); };
    auto s0_a = [&](int m0, int k0) {
        const float *x = S0f + (m0 + g) * OS + k0 + 2 * q;
        return make_a(ld2(x), ld2(x + 8 * OS), ld2(x + 8), ld2(x + 8 * OS + 8));
    };
    auto s0_at = [&](int m0, int k0) {
        const float *x = S0f + (k0 + 2 * q) * OS + m0 + g;
        return make_a(make_float2(x[0], x[OS]), make_float2(x[8], x[OS + 8]), make_float2(x[8 * OS], x[9 * OS]),
                      make_float2(x[8 * OS + 8], x[9 * OS + 8]));
    };
    const float *FC = reinterpret_cast<const float *>(Bs + oQQ);  // factor block of the current chunk
    auto stage_fac = [&](int c) {
        if constexpr (kFac) {
            if (ccopy == 7) bulk_g2s(Bs + oQQ, p.fac_in + ((size_t)bh * nchunks + c) * fac::kWords, kFacWords * 4, &bar);
        }
    };
    stage_in(nchunks - 1);
    stage_fac(nchunks - 1);
    if (tid == 0) mbar_arrive(&bar);

    for (int c = nchunks - 1; c >= 0; --c) {
        const int t0 = c * C;
        const int nv = min(C, p.T - t0);
        const bool last = c == nchunks - 1;
        const unsigned ph = (nchunks - 1 - c) & 1;
        mbar_wait(&bar, ph, p.err, &lost);
        if (tid == 0 && c > 0) mbar_expect_tx(&bar, kChunkBytes + (last ? kPhantomTx : 0u));
        // The last chunk's gradient stores must have read their staging before the
        // start state lands in the S_0 slot (dr, dw, dk, dv: lanes 0..3 of warp 0)
        // and before the v split and SA, both after a later block barrier, overwrite
        // the v and SA slots (da, db: lanes 0..1 of warp 1).  Each issuing lane waits
        // for its own store after the first splits.
        auto drain_then_load_s0 = [&]() {
            if (warp == 1 && lane < 2) bulk_wait_read();
            if (warp == 0) {
                if (lane < 4) bulk_wait_read();
                __syncwarp();
                if (lane == 0) {
                    load_s0(c);
                    // the next start state into L2 now, so that its copy at the next
                    // chunk start does not wait on DRAM
                    if (c > 0) tma_prefetch_2d(&maps.m[7], (bh * p.nck + c - 1) * 64);
                }
            }
        };
        // dy split into [t][i] quads; it needs no decay: with plain inputs warps 0 and 1 split it
        // while warps 2 and 3 form the decays, with the producers (all four warps form the decays)
        // or the epilogue (dy is the converted do) every warp splits it after the decays
        auto split_dy = [&](int e) {
            const int t = e >> 4, j = (e & 15) * 4;
            st_hl4(hi_of(Bs, oDYH), lo_of(Bs, oDYH, 16), t, j, *reinterpret_cast<const float4 *>(dyf + t * SP + j));
        };
        if constexpr (!kP && !kGN) {
            if (warp < 2) {
#pragma unroll
                for (int m = 0; m < 4; ++m) split_dy(tid + 64 * m);
            }
        }
        // the cumulative decays on warps 2 and 3 (warps 0 and 1 have just issued the gradient stores)
        const bool exact = __syncthreads_or(prep_decay<kP, E, !kP>(raw, dd, nv, 64, kP ? sgs : nullptr));
        if (lost) {  // every thread has passed its wait (the barrier above): leave together
            stuck = c;
            break;
        }
        if constexpr (kGN) {  // do -> dy through the epilogue: 16 lanes per token (four channels each),
                              // two tokens per warp at a time; every sum in one round of four shuffle levels
            const int j = 4 * (lane & 15);
            const float4 gw = *reinterpret_cast<const float4 *>(gnp + j);
            const float4 rk = *reinterpret_cast<const float4 *>(gnp + 64 + j);
            auto sum16 = [](float x) {
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                return x;
            };
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 4 * warp + 2 * u + (lane >> 4);
                const float4 y4 = *reinterpret_cast<const float4 *>(Gm + t * SP + j);
                const float4 d4 = *reinterpret_cast<const float4 *>(dyf + t * SP + j);
                const float4 v4 = ld_raw4(raw, VV, t, j), r4 = ld_raw4(raw, VR, t, j), k4 = ld_raw4(raw, VK, t, j);
                const float dn[4] = {d4.x * gw.x, d4.y * gw.y, d4.z * gw.z, d4.w * gw.w};
                // one round of sums, about a shift m0 (the token's first channel) so that the
                // moments of y - m0 do not cancel: mean = m0 + E[z], var = E[z^2] - E[z]^2,
                // sum(dn (y - mean)) = sum(dn z) - E[z] sum(dn)
                const float m0 = __shfl_sync(0xffffffffu, y4.x, lane & 16);
                const float z[4] = {y4.x - m0, y4.y - m0, y4.z - m0, y4.w - m0};
                const float sz = sum16(z[0] + z[1] + z[2] + z[3]);
                const float szz = sum16(z[0] * z[0] + z[1] * z[1] + z[2] * z[2] + z[3] * z[3]);
                const float sdn = sum16(dn[0] + dn[1] + dn[2] + dn[3]);
                const float sdz = sum16(dn[0] * z[0] + dn[1] * z[1] + dn[2] * z[2] + dn[3] * z[3]);
                const float sb = sum16(r4.x * k4.x * rk.x + r4.y * k4.y * rk.y + r4.z * k4.z * rk.z + r4.w * k4.w * rk.w);
                const float ds = sum16(d4.x * v4.x + d4.y * v4.y + d4.z * v4.z + d4.w * v4.w);
                const float ez = sz * (1.f / 64.f);
                const float var = fmaxf(szz * (1.f / 64.f) - ez * ez, 0.f);
                const float c[4] = {z[0] - ez, z[1] - ez, z[2] - ez, z[3] - ez};
                const float rstd = rsqrtf(var + kGnEps);
                const float mn = sdn * (1.f / 64.f), mx = rstd * (sdz - ez * sdn) * (1.f / 64.f);
                float x[4], dy[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[i] = c[i] * rstd;
                    dy[i] = rstd * (dn[i] - mn - x[i] * mx);
                }
                *reinterpret_cast<float4 *>(dyf + t * SP + j) = make_float4(dy[0], dy[1], dy[2], dy[3]);
                *reinterpret_cast<float4 *>(Gm + t * SP + j) = make_float4(d4.x * sb, d4.y * sb, d4.z * sb, d4.w * sb);
                if ((lane & 15) == 0) dsv[t] = ds;
                pgw.x += d4.x * x[0]; pgw.y += d4.y * x[1]; pgw.z += d4.z * x[2]; pgw.w += d4.w * x[3];
                pgb.x += d4.x; pgb.y += d4.y; pgb.z += d4.z; pgb.w += d4.w;
                prk.x += ds * r4.x * k4.x; prk.y += ds * r4.y * k4.y; prk.z += ds * r4.z * k4.z; prk.w += ds * r4.w * k4.w;
            }
            __syncthreads();
        }
        if (exact) {
            if constexpr (kSO) {
                bwd_chunk_exact_state<E, kP>(raw, dyf, Gh, nv);
                __syncthreads();  // every lane has read the chunk's rows before the copies refill them
            } else {
                drain_then_load_s0();
                mbar_wait(&bar_s, ph, p.err, &lost);
                bwd_chunk_exact<E, kP, OS, kGN>(raw, dyf, S0f, reinterpret_cast<float *>(Bs + B_BT),
                                                reinterpret_cast<float *>(Bs + B_Y), Gh, nv, p, base0, tstride, t0,
                                                carryA, carryB, Gm, dsv, p.r_k + h * 64);
                fence_proxy_async();  // the per-token path wrote into slots the copies refill
                __syncthreads();
            }
            if (c > 0) {
                stage_in(c - 1);
                stage_fac(c - 1);
                if (tid == 0) mbar_arrive(&bar);
            }
            continue;
        }
        const float *dC = dd + (C - 1) * DS;
        // (G diag(d_C)) as the A fragment of key columns 16 kk .. 16 kk + 15 (this warp's value rows)
        auto gd_a = [&](int kk) {
            const float2 d0 = *reinterpret_cast<const float2 *>(dC + 16 * kk + 2 * q);
            const float2 d1 = *reinterpret_cast<const float2 *>(dC + 16 * kk + 8 + 2 * q);
            return make_a(make_float2(Gh[2 * kk][0] * d0.x, Gh[2 * kk][1] * d0.y),
                          make_float2(Gh[2 * kk][2] * d0.x, Gh[2 * kk][3] * d0.y),
                          make_float2(Gh[2 * kk + 1][0] * d1.x, Gh[2 * kk + 1][1] * d1.y),
                          make_float2(Gh[2 * kk + 1][2] * d1.x, Gh[2 * kk + 1][3] * d1.y));
        };
        // G5: G_prev = G diag(d_C) + [DY | DSA] [R^ | A^]^T  (rows = value index)
        auto g5 = [&](const AFrag &dyA, const AFrag &dsA) {
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                BFrag rr[2], aa[2];
                ldb2_t(RH, 16 * pp, 0, lane, rr[0], rr[1]);
                ldb2_t(AH, 16 * pp, 0, lane, aa[0], aa[1]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * pp + u;
                    const float2 dc = *reinterpret_cast<const float2 *>(dC + 8 * nt + 2 * q);
                    Gh[nt][0] *= dc.x; Gh[nt][1] *= dc.y; Gh[nt][2] *= dc.x; Gh[nt][3] *= dc.y;
                }
                mma3n<2>(Gh + 2 * pp, dyA, rr);
                mma3n<2>(Gh + 2 * pp, dsA, aa);
            }
        };

        // ================= split every operand matrix once (S_0 is split where it is read)
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // decay-scaled vectors: [t][j] quads
            // with the factor cache, warp w converts its own 16-key slab (all
            // tokens); the block barrier after the splits shows every slab to G2
            const int e = kFac ? lane + 32 * m : tid + NT * m;
            const int t = kFac ? slab_token(e) : e >> 4, j = kFac ? 16 * warp + (e & 3) * 4 : (e & 15) * 4;
            const float4 d = *reinterpret_cast<const float4 *>(dd + t * DS + j);
            const float4 dp = t ? *reinterpret_cast<const float4 *>(dd + (t - 1) * DS + j) : make_float4(1.f, 1.f, 1.f, 1.f);
            const float4 id = rcp4(d);
            st_hl4(hi_of(Bs, oBT), lo_of(Bs, oBT, 16), t, j, mul4(in_b4<kP>(raw, t, j), id));
            if constexpr (kP) *reinterpret_cast<float4 *>(avs + t * OS + j) = ld_raw4(raw, VB, t, j);
            if constexpr (!kSO) st_hl4(hi_of(Bs, B_KT), lo_of(Bs, B_KT, 16), t, j, mul4(ld_raw4(raw, VK, t, j), id));
            st_hl4(hi_of(Bs, oAH), lo_of(Bs, oAH, 16), t, j, mul4(in_a4<kP>(raw, t, j), dp));
            st_hl4(hi_of(Bs, oRH), lo_of(Bs, oRH, 16), t, j, mul4(ld_raw4(raw, VR, t, j), d));
        }
        if constexpr (kP || kGN) {
#pragma unroll
            for (int m = 0; m < 2; ++m) split_dy(tid + NT * m);
        }
        if constexpr (!kSO) drain_then_load_s0();
        if constexpr (kFac)
            __syncwarp();
        else
            __syncthreads();

        // ================= per-chunk operands (no state involved)
        if constexpr (!kFac) {
        {   // Gram [B~; K~] [A^; R^]^T: warp -> m-tile (b~ | k~), n-tile pair (a^ | r^)
            const int mt = warp >> 1;
            float acc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const AFrag af = lda(mt ? KT : BT, 0, 16 * kk, lane);
                BFrag b0, b1;
                ldb2((warp & 1) ? RH : AH, 0, 16 * kk, lane, b0, b1);
                const BFrag bq[2] = {b0, b1};
                mma3n<2>(acc, af, bq);
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
        prep_inverse(Gm, Wm);
        __syncthreads();
        // A' = W^T-weighted A^ (M = token, N = key): warp 0 keys 0..31, warps 2 and 3
        // keys 16w..16w+15 (warp 3 also W Q_b); warp 1 builds M_k' and then Q'
        auto qbv = [&](int u, int t) { return u <= t ? Gm[u * GS + 16 + t] : 0.f; };
        if (warp != 1) {
            const AFrag wt = make_a(make_float2(Wm[(2 * q) * WS + g], Wm[(2 * q + 1) * WS + g]),
                                    make_float2(Wm[(2 * q) * WS + g + 8], Wm[(2 * q + 1) * WS + g + 8]),
                                    make_float2(Wm[(2 * q + 8) * WS + g], Wm[(2 * q + 9) * WS + g]),
                                    make_float2(Wm[(2 * q + 8) * WS + g + 8], Wm[(2 * q + 9) * WS + g + 8]));
            if (warp == 0)
                build_ap<2>(wt, AH, Bs, 0, lane);
            else
                build_ap<1>(wt, AH, Bs, warp, lane);
        }
        if (warp == 3) {  // W Q_b -> rows 16..31 of the [Q'; W Q_b] block
            const AFrag wa = make_a(make_float2(Wm[g * WS + 2 * q], Wm[g * WS + 2 * q + 1]),
                                    make_float2(Wm[(g + 8) * WS + 2 * q], Wm[(g + 8) * WS + 2 * q + 1]),
                                    make_float2(Wm[g * WS + 2 * q + 8], Wm[g * WS + 2 * q + 9]),
                                    make_float2(Wm[(g + 8) * WS + 2 * q + 8], Wm[(g + 8) * WS + 2 * q + 9]));
            __nv_bfloat16 *qh = hi_of(Bs, B_QQ), *ql = lo_of(Bs, B_QQ, 32);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tc = 8 * nt + 2 * q, t = 8 * nt + g;
                float cb[4] = {0.f, 0.f, 0.f, 0.f};
                mma3(cb, wa, make_b(make_float2(qbv(2 * q, t), qbv(2 * q + 1, t)),
                                    make_float2(qbv(2 * q + 8, t), qbv(2 * q + 9, t))));
                st_hl(qh, ql, 16 + g, tc, cb[0], cb[1]);  // (W Q_b)[t][s]
                st_hl(qh, ql, 24 + g, tc, cb[2], cb[3]);
            }
        }
        if (warp == 1) {  // M_k' = M_k W, then Q' = Q_k + M_k' Q_b (16 x 16)
            auto mk = [&](int s, int u) { return u > s ? Gm[(16 + s) * GS + u] : 0.f; };
            auto qkv = [&](int s, int t) { return s <= t ? Gm[(16 + s) * GS + 16 + t] : 0.f; };
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
            float cq[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tc = 8 * nt + 2 * q, t = 8 * nt + g;
                cq[nt][0] = qkv(g, tc); cq[nt][1] = qkv(g, tc + 1); cq[nt][2] = qkv(g + 8, tc); cq[nt][3] = qkv(g + 8, tc + 1);
                mma3(cq[nt], amp, make_b(make_float2(qbv(2 * q, t), qbv(2 * q + 1, t)),
                                         make_float2(qbv(2 * q + 8, t), qbv(2 * q + 9, t))));
            }
            __nv_bfloat16 *mh = hi_of(Bs, B_MK), *ml = lo_of(Bs, B_MK, 16);
            __nv_bfloat16 *qh = hi_of(Bs, B_QQ), *ql = lo_of(Bs, B_QQ, 32);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tc = 8 * nt + 2 * q;
                st_hl(mh, ml, g, tc, cm[nt][0], cm[nt][1]);  // M_k'[s][t]
                st_hl(mh, ml, g + 8, tc, cm[nt][2], cm[nt][3]);
                st_hl(qh, ql, g, tc, cq[nt][0], cq[nt][1]);  // Q'[t][s]
                st_hl(qh, ql, g + 8, tc, cq[nt][2], cq[nt][3]);
            }
        }
        __syncthreads();
        }
        __syncthreads();  // every b~ / k~ slab is split; warp 0 has drained the gradient stores
        if constexpr (kSO) {  // X_B = (G diag(d_C)) B~^T, DSA = X_B W^T + DY (W Q_b)^T, then G5
            float xbs[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const AFrag gf = gd_a(kk);
                BFrag bq[2];
                ldb2(BT, 0, 16 * kk, lane, bq[0], bq[1]);
                mma3n<2>(xbs, gf, bq);
            }
            const AFrag awn = ld_afrag(FC + fac::kWA, lane), xb = a_from_acc(xbs, 0);
            float dsb[2][4] = {};
            { const BFrag bw[2] = {tb(awn, 0), tb(awn, 1)}; mma3n<2>(dsb, xb, bw); }
            const AFrag dyA = lda_t(DYH, 16 * warp, 0, lane);
            {
                BFrag bq[2];
                ld_bfrags(FC + fac::kWQbB, lane, bq[0], bq[1]);
                mma3n<2>(dsb, dyA, bq);
            }
            const AFrag dsA = a_from_acc(dsb, 0);
            __syncthreads();  // the chunk's rows, dy and factors are read
            if (c > 0) {
                stage_in(c - 1);
                stage_fac(c - 1);
                if (tid == 0) mbar_arrive(&bar);
            }
            g5(dyA, dsA);
            __syncthreads();  // G5 has read d_C, r^ and a^ before the next chunk's decays and splits
            continue;
        }
        // v split: warp w its own 16 value columns (all tokens), which is all its vA
        // reads; the other readers come after the barrier that follows G2
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int e = lane + 32 * m, t = slab_token(e), i = 16 * warp + (e & 3) * 4;
            st_hl4(hi_of(Bs, B_VV), lo_of(Bs, B_VV, 16), t, i, ld_raw4(raw, VV, t, i));
        }
        __syncwarp();

        // ================= state-dependent products
        // G1: SA = S_0 A' + V M_k'  (rows = value index)
        float sa[2][4] = {};
        const AFrag vA = lda_t(VM, 16 * warp, 0, lane);
        if constexpr (kFac) {  // SA from the forward
            ld_acc2(FC + fac::kSA + 256 * warp, sa[0], sa[1], lane);
        } else {
            mbar_wait(&bar_s, ph, p.err, &lost);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const AFrag sf = s0_a(16 * warp, 16 * kk);
                BFrag b0, b1;
                ldb2(AP, 0, 16 * kk, lane, b0, b1);
                mma3(sa[0], sf, b0);
                mma3(sa[1], sf, b1);
            }
            BFrag b0, b1;
            ldb2_t(MK, 0, 0, lane, b0, b1);
            mma3(sa[0], vA, b0);
            mma3(sa[1], vA, b1);
        }
        {
            __nv_bfloat16 *shh = hi_of(Bs, B_SAH), *shl = lo_of(Bs, B_SAH, 16);
            st_acc_t16(shh, shl, 0, 16 * warp, sa, lane);  // SA[i][t] -> SAH[t][i]
        }

        // the dw running sum starts at diag(dsT^T sT): sT from the last chunk's start state
        if (last && p.dsT) {
            mbar_wait(&bar_s, ph, p.err, &lost);
            const AFrag saA = make_a(make_float2(sa[0][0], sa[0][1]), make_float2(sa[0][2], sa[0][3]),
                                     make_float2(sa[1][0], sa[1][1]), make_float2(sa[1][2], sa[1][3]));
            float part[8][2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                BFrag bb0, bb1, kb0, kb1;
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {  // n-tile pairs 4*half + 2*pp
                    const int n0 = 32 * half + 16 * pp;
                    ldb2_t(BT, n0, 0, lane, bb0, bb1);
                    ldb2_t(KT, n0, 0, lane, kb0, kb1);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int nt = 4 * half + 2 * pp + u, j0 = 8 * nt + 2 * q;
                        const float2 x = ld2(S0f + rA * OS + j0), z = ld2(S0f + rB * OS + j0);
                        float ST[4] = {x.x, x.y, z.x, z.y};
                        mma3(ST, saA, u ? bb1 : bb0);
                        mma3(ST, vA, u ? kb1 : kb0);
                        const float2 dc = *reinterpret_cast<const float2 *>(dC + j0);
                        ST[0] *= dc.x; ST[1] *= dc.y; ST[2] *= dc.x; ST[3] *= dc.y;
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            part[nt][e] = rows_sum(__fmaf_rn(Gh[nt][e], ST[e], __fmul_rn(Gh[nt][2 + e], ST[2 + e])));
                    }
                }
            }
            // the Gram slot is idle between W and Gam: 4 x 64 floats of per-warp column sums
            if (g == 0) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    carp[warp * 64 + 8 * nt + 2 * q] = part[nt][0];
                    carp[warp * 64 + 8 * nt + 2 * q + 1] = part[nt][1];
                }
            }
            __syncthreads();
            carryA = carp[rA] + carp[64 + rA] + carp[128 + rA] + carp[192 + rA];
            carryB = carp[rB] + carp[64 + rB] + carp[128 + rB] + carp[192 + rB];
        }

        // G2: [DV | DSA] = G [K' | B'] + DY [Q'^T | (W Q_b)^T], with K' = d_C o (K~ + M_k' B~) and
        // B' = d_C o (W B~) never formed: X = (G diag(d_C)) [K~ | B~]^T, then
        //   G K'^T = X_K + X_B M_k'^T,   G B'^T = X_B W^T   (16 x 16 products on this warp's rows)
        float dvs[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag gf = gd_a(kk);
            BFrag b0, b1, b2, b3;
            ldb2(KT, 0, 16 * kk, lane, b0, b1);
            ldb2(BT, 0, 16 * kk, lane, b2, b3);
            { const BFrag bq[4] = {b0, b1, b2, b3}; mma3n<4>(dvs, gf, bq); }
        }
        {
            // M_k' (M = token t, K = s) and W as A fragments, their transposes' B fragments by tb
            AFrag amk, awn;
            if constexpr (kFac) {
                amk = ld_afrag(FC + fac::kMkA, lane);
                awn = ld_afrag(FC + fac::kWA, lane);
            } else {
                amk = lda(MK, 0, 0, lane);
                awn = make_a(make_float2(Wm[g * WS + 2 * q], Wm[g * WS + 2 * q + 1]),
                             make_float2(Wm[(g + 8) * WS + 2 * q], Wm[(g + 8) * WS + 2 * q + 1]),
                             make_float2(Wm[g * WS + 2 * q + 8], Wm[g * WS + 2 * q + 9]),
                             make_float2(Wm[(g + 8) * WS + 2 * q + 8], Wm[(g + 8) * WS + 2 * q + 9]));
            }
            const AFrag xb = a_from_acc(dvs, 1);  // X_B (tiles 2, 3)
            float dsa[2][4] = {};
            { const BFrag bm[2] = {tb(amk, 0), tb(amk, 1)}; mma3n<2>(dvs, xb, bm); }
            { const BFrag bw[2] = {tb(awn, 0), tb(awn, 1)}; mma3n<2>(dsa, xb, bw); }
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) dvs[2 + u][e] = dsa[u][e];
        }
        const AFrag dyA = lda_t(DYH, 16 * warp, 0, lane);
        {
            BFrag b0, b1, b2, b3;
            if constexpr (kFac) {
                ld_bfrags(FC + fac::kQB, lane, b0, b1);
                ld_bfrags(FC + fac::kWQbB, lane, b2, b3);
            } else {
                ldb2(QQ, 0, 0, lane, b0, b1);
                ldb2(QQ, 16, 0, lane, b2, b3);
            }
            { const BFrag bq[4] = {b0, b1, b2, b3}; mma3n<4>(dvs, dyA, bq); }
        }
        if constexpr (kGN) {  // + the bonus's own dv, do s, from the y slot (before the next copies refill it)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t = 8 * nt + 2 * q;
                dvs[nt][0] += Gm[t * SP + rA];
                dvs[nt][1] += Gm[(t + 1) * SP + rA];
                dvs[nt][2] += Gm[t * SP + rB];
                dvs[nt][3] += Gm[(t + 1) * SP + rB];
            }
        }
        {
            __nv_bfloat16 *dhh = hi_of(Bs, B_DSH), *dhl = lo_of(Bs, B_DSH, 16);
            st_acc_t16(dhh, dhl, 0, 16 * warp, dvs + 2, lane);  // DSA[i][t] -> DSH[t][i]
        }
        const AFrag dsA = make_a(make_float2(dvs[2][0], dvs[2][1]), make_float2(dvs[2][2], dvs[2][3]),
                                 make_float2(dvs[3][0], dvs[3][1]), make_float2(dvs[3][2], dvs[3][3]));
        // kP: -0.606531 sigmoid (1 - sigmoid) of w_pre at this lane's dw positions (key rows rA / rB,
        // tokens 2q, 2q + 1, 8 + 2q, 9 + 2q), from the sigmoid of w_pre itself that the decay
        // phase kept (before G3 writes M4 over it): recovering the sigmoid from the decays
        // (-ln(w) / 0.606531) would lose its relative precision where it is small (w rounds to 1)
        float sgf[2][4];
        if constexpr (kP) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = 8 * (m >> 1) + 2 * q + (m & 1);
                    const float sg = sgs[t * DS + (hr ? rB : rA)];
                    sgf[hr][m] = -kDecayScale * sg * (1.f - sg);
                }
        }
        __syncthreads();
        if (c > 0) {  // this chunk's inputs, dy and factors are consumed: fetch the previous chunk's
            stage_in(c - 1);
            stage_fac(c - 1);
            if (tid == 0) mbar_arrive(&bar);
        }

        // G3: [DR | DA] (rows = key index j = rA / rB)
        float x3[4][4] = {};
        {   // Gam = [SA | V]^T [DY | DSA] (32 x 32): warp -> m-tile (SA | V), n-tile pair (DY | DSA),
            // written straight into its two masked split blocks:
            //   M3[k][n] = Gam[k][n] where (n < 16 ? s <= t : s < t)           (s = k % 16, t = n % 16)
            //   M4[k][n] = Gam[n < 16 ? 16 + t : t][k] where (k < 16 ? s >= t : s > t)
            // M3 pairs (b~_s | k~_s) with (dy_t | dsa_t); M4 pairs (r^_s | a^_s) with (v_t | sa_t)
            // G3's S_0 part, S_0^T [DY | DSA], needs only DY, DSA and S_0: it shares
            // this loop (and its DY / DSA fragments) with Gam.
            const int mt = warp >> 1;
            float acc[2][4] = {};
            mbar_wait(&bar_s, ph, p.err, &lost);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                BFrag bq[4];
                ldb2(DYH, 0, 16 * kk, lane, bq[0], bq[1]);
                ldb2(DSH, 0, 16 * kk, lane, bq[2], bq[3]);
                // v rows: with bf16 inputs their lo part is zero and is not loaded
                const AFrag af = (mt && !kVLo) ? lda_hi(VM, 0, 16 * kk, lane) : lda(mt ? VM : SAH, 0, 16 * kk, lane);
                const bool ds = warp & 1;
                const BFrag gq[2] = {ds ? bq[2] : bq[0], ds ? bq[3] : bq[1]};
                mma3n<2>(acc, af, gq);
                const AFrag sT = s0_at(16 * warp, 16 * kk);
                mma3n<4>(x3, sT, bq);
            }
            __nv_bfloat16 *h3 = hi_of(Bs, B_M3), *l3 = lo_of(Bs, B_M3, 32);
            __nv_bfloat16 *h4 = hi_of(Bs, B_M4), *l4 = lo_of(Bs, B_M4, 32);
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
            st_acc16(h3, l3, 16 * mt, 16 * (warp & 1), m3, lane);
            // M4[n][nn] with n = the Gam column, nn = the Gam row with its halves swapped
            st_acc_t16(h4, l4, 16 * (warp & 1), mt ? 0 : 16, m4, lane);
        }

        __syncthreads();  // masked Gam blocks visible; S_0, dy and DSA no longer read
        // b~ and k~ of this warp's key rows as A operands, kept for the outputs
        const AFrag btA = lda_t(BT, 16 * warp, 0, lane), ktA = lda_t(KT, 16 * warp, 0, lane);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            BFrag bq[4];
            ldb2_t(M3, 0, 16 * kk, lane, bq[0], bq[1]);
            ldb2_t(M3, 16, 16 * kk, lane, bq[2], bq[3]);
            mma3n<4>(x3, kk ? ktA : btA, bq);
        }
        // the S_0 slot takes G d_C (split)
        {
            __nv_bfloat16 *gh = hi_of(Bs, B_SX), *gl = lo_of(Bs, B_SX, 64);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                float gd[2][4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * pp + u;
                    const float2 dc = *reinterpret_cast<const float2 *>(dC + 8 * nt + 2 * q);
                    gd[u][0] = Gh[nt][0] * dc.x; gd[u][1] = Gh[nt][1] * dc.y;
                    gd[u][2] = Gh[nt][2] * dc.x; gd[u][3] = Gh[nt][3] * dc.y;
                }
                st_acc16(gh, gl, 16 * warp, 16 * pp, gd, lane);
            }
        }
        __syncthreads();  // G d_C visible

        // G4: [DK | DB] (rows = key index)
        float x4[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const AFrag gT = lda_t(SX, 16 * warp, 16 * kk, lane);
            BFrag b0, b1, b2, b3;
            if constexpr (kVLo)
                ldb2(VM, 0, 16 * kk, lane, b0, b1);
            else
                ldb2_hi(VM, 0, 16 * kk, lane, b0, b1);
            ldb2(SAH, 0, 16 * kk, lane, b2, b3);
            {
                const BFrag bv[2] = {b0, b1}, bs[2] = {b2, b3};
                mma3n<2, true, kVLo>(x4, gT, bv);
                mma3n<2>(x4 + 2, gT, bs);
            }
        }
        const AFrag rhA = lda_t(RH, 16 * warp, 0, lane), ahA = lda_t(AH, 16 * warp, 0, lane);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            BFrag bq[4];
            ldb2_t(M4, 0, 16 * kk, lane, bq[0], bq[1]);
            ldb2_t(M4, 16, 16 * kk, lane, bq[2], bq[3]);
            mma3n<4>(x4, kk ? ahA : rhA, bq);
        }

        // G5, issued before the output code so that its MMAs run under the scalar work
        g5(dyA, dsA);
        // ================= gradients: staged as [t][key] tiles (stride OS) in the
        // S_0 / G d_C quarters and the v and SA slots, then one tensor store each
        __syncthreads();  // G4 and G5 no longer read those slots
        float *const gdr = reinterpret_cast<float *>(Bs + B_SX), *const gdw = gdr + 1152, *const gdk = gdr + 2 * 1152;
        float *const gdv = gdr + 3 * 1152, *const gda = reinterpret_cast<float *>(Bs + B_VV);
        float *const gdb = reinterpret_cast<float *>(Bs + B_SAH);
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
                    if constexpr (kGN) {  // + the bonus's dr = ds k r_k and dk = ds r r_k
                        const float rkr = m < 2 ? rkA : rkB;
                        gdr[t * OS + row] = d * xr + dsv[t] * (kv[vi] * d) * rkr;
                        gdk[t * OS + row] = inv * xk + dsv[t] * (rv[vi] * inv) * rkr;
                    } else {
                        gdr[t * OS + row] = d * xr;
                        gdk[t * OS + row] = inv * xk;
                    }
                    if constexpr (kP) {  // dkk = -da + avec db, davec = kk db (k_comp_keymod)
                        const float db_ = inv * xb;
                        gda[t * OS + row] = avs[t * OS + row] * db_ - dp * xa;
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
        // from lanes 0..1 of warp 1 (the two warps issue theirs side by side)
        const int o = warp == 0 ? lane : warp == 1 ? 4 + lane : 6;
        if ((warp == 0 && lane < 4) || (warp == 1 && lane < 2)) {
            const float *const tile = o < 4 ? gdr + 1152 * o : o == 4 ? gda : gdb;
            tma_store_rows(&omaps.m[o], tile, h, t0, bi);
            bulk_commit();
        }
    }
    if ((warp == 0 && lane < 4) || (warp == 1 && lane < 2)) bulk_wait_all();
    if (stuck >= 0) {
        mbar_drain(&bar, (nchunks - 1 - stuck) & 1);
        if (tid == 0 && s_phase >= 0) mbar_drain(&bar_s, s_phase);
    }
    if constexpr (kGN) {  // this head's parameter-gradient sums: both half-warps, then the four warps
        float4 *const acc3[3] = {&pgw, &pgb, &prk};
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            float4 &v = *acc3[a];
            v.x += __shfl_xor_sync(0xffffffffu, v.x, 16);
            v.y += __shfl_xor_sync(0xffffffffu, v.y, 16);
            v.z += __shfl_xor_sync(0xffffffffu, v.z, 16);
            v.w += __shfl_xor_sync(0xffffffffu, v.w, 16);
        }
        __syncthreads();
        float *const sc = Gm;  // [warp][3][64]
        if (lane < 16) {
            *reinterpret_cast<float4 *>(sc + (warp * 3 + 0) * 64 + 4 * lane) = pgw;
            *reinterpret_cast<float4 *>(sc + (warp * 3 + 1) * 64 + 4 * lane) = pgb;
            *reinterpret_cast<float4 *>(sc + (warp * 3 + 2) * 64 + 4 * lane) = prk;
        }
        __syncthreads();
        for (int o = tid; o < 3 * 64; o += NT)
            p.gn_part[(size_t)bh * 192 + o] = sc[o] + sc[192 + o] + sc[384 + o] + sc[576 + o];
    }
    if (p.ds0) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<float2 *>(p.ds0 + sbase + rA * 64 + 8 * nt + 2 * q) = make_float2(Gh[nt][0], Gh[nt][1]);
            *reinterpret_cast<float2 *>(p.ds0 + sbase + rB * 64 + 8 * nt + 2 * q) = make_float2(Gh[nt][2], Gh[nt][3]);
        }
    }
}

template <typename E, bool kFac, bool kP, bool kGN = false, bool kSO = false>
cudaError_t launch_t(const SeqArgs &p, cudaStream_t st) {
    const size_t sm = bwd_smem_bytes<E, kSO, kGN>();
    InputMaps maps{};
    OutputMaps omaps{};
    cudaError_t e = encode_input_maps(&maps, p, p.dy);  // six inputs, dy (or do), and the checkpoints (box OS x 64)
    // the state-gradient pass reads no checkpoint and stores no per-token gradient
    if (e == cudaSuccess && !kSO) e = encode_ckpt_map(&maps.m[7], p.ckpt_in, (long long)p.B * p.H * p.nck * 64, 64);
    if (e == cudaSuccess && kGN) e = encode_rows_map(&maps.m[8], p.y_in, 4, p.B, p.T, p.H);  // the forward's y
    if (e == cudaSuccess && !kSO) e = encode_output_maps(&omaps, p);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(wkv7_bwd_chunk_kernel<E, kFac, kP, kGN, kSO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
    if (e != cudaSuccess) return e;
    wkv7_bwd_chunk_kernel<E, kFac, kP, kGN, kSO><<<p.B * p.H, NT, sm, st>>>(p, maps, omaps);
    return cudaGetLastError();
}

// Sum of the per-(b,h) parameter-gradient partials over the batch rows, in a
// fixed order (no atomics): one thread per (h, parameter, channel).
__global__ void wkv7_gn_param_reduce_kernel(int B, int H, const float *part, float *dgn_w, float *dgn_b, float *dr_k) {
    const int h = blockIdx.x, o = threadIdx.x;  // o = parameter * 64 + channel
    float s = 0.f;
    for (int b = 0; b < B; ++b) s += part[((size_t)b * H + h) * 192 + o];
    float *const dst[3] = {dgn_w, dgn_b, dr_k};
    dst[o >> 6][h * 64 + (o & 63)] = s;
}

}  // namespace

bool backward_chunk_supported(const SeqArgs &p) { return p.L == C; }

// With the factor cache, the backward can run the two 64-row state products
// that feed only the gradient outputs on the fifth-generation tensor cores
// (wkv7_chunk_bwd_tc.cu); WKV7_BACKWARD_KERNEL=tcgen05 in the environment
// (read at each launch) selects that kernel, "mma" or nothing this file's.
// The warp-level kernel is the default: on the bf16 B=16 T=4096 H=32 workload
// (two CTAs per SM) it measured 2.44 ms against 3.17 ms.
static bool tensor_core_backward() {
    const char *v = getenv("WKV7_BACKWARD_KERNEL");
    return v && strcmp(v, "tcgen05") == 0;
}

cudaError_t launch_gn_param_reduce(int B, int H, const float *part, float *dgn_w, float *dgn_b, float *dr_k,
                                   cudaStream_t st) {
    wkv7_gn_param_reduce_kernel<<<H, 192, 0, st>>>(B, H, part, dgn_w, dgn_b, dr_k);
    return cudaGetLastError();
}

cudaError_t launch_backward_chunk(const SeqArgs &p, cudaStream_t st) {
    if (p.gn_w) {  // the output epilogue's backward in front: factor-cache path, no fused producers
        if (!p.fac_in || p.prod) return cudaErrorInvalidValue;
        return p.dtype == 1 ? launch_t<__nv_bfloat16, true, false, true>(p, st) : launch_t<float, true, false, true>(p, st);
    }
    if (backward_tc_supported(p) && tensor_core_backward()) return launch_backward_tc(p, st);
    if (p.prod) {  // the fused producers run with the factor cache only
        if (!p.fac_in) return cudaErrorInvalidValue;
        return p.dtype == 1 ? launch_t<__nv_bfloat16, true, true>(p, st) : launch_t<float, true, true>(p, st);
    }
    if (p.fac_in) return p.dtype == 1 ? launch_t<__nv_bfloat16, true, false>(p, st) : launch_t<float, true, false>(p, st);
    return p.dtype == 1 ? launch_t<__nv_bfloat16, false, false>(p, st) : launch_t<float, false, false>(p, st);
}

cudaError_t launch_backward_state(const SeqArgs &p, cudaStream_t st) {
    if (!p.fac_in || !p.ds0 || p.prod || p.gn_w || p.L != C) return cudaErrorInvalidValue;
    return p.dtype == 1 ? launch_t<__nv_bfloat16, true, false, false, true>(p, st)
                        : launch_t<float, true, false, false, true>(p, st);
}

}  // namespace wkv7
