// Shared pieces of the chunked WKV7 kernels (forward and backward): TMA
// staging of a chunk on an mbarrier, the cumulative decays of a chunk and the
// inverse W = (I - M_b)^{-1}.
//
// Notation (one (b,h), one chunk of C = 16 tokens, local index t = 0..15):
//   d_t  = w_0 o ... o w_t          cumulative decay per key column
//   a^_t = a_t o d_{t-1}            r^_t = r_t o d_t
//   b~_t = b_t / d_t                k~_t = k_t / d_t
//   Gram rows (b~_s, k~_s), columns (a^_t, r^_t):
//     M_b[s][t] = b~_s.a^_t  (s<t)   M_k[s][t] = k~_s.a^_t  (s<t)
//     Q_b[s][t] = b~_s.r^_t  (s<=t)  Q_k[s][t] = k~_s.r^_t  (s<=t)
// The unrolled recurrence of a chunk is
//   S_t = (S_0 + sum_{s<=t} sa_s b~_s^T + v_s k~_s^T) diag(d_t),
//   sa_t = S_0 a^_t + sum_{s<t} sa_s M_b[s][t] + v_s M_k[s][t].
#pragma once
#include <cuda.h>

#include "wkv7_internal.cuh"
#include "wkv7_mma.cuh"

namespace wkv7 {
namespace chunk {

constexpr int C = 16;          // tokens per chunk
constexpr int SP = 72;         // row stride (floats) of [token][64] and [row][64] arrays
constexpr int DS = 68;         // row stride (floats) of the cumulative decays d[t][j]: reads at
                               // tokens 2q, 2q + 1 and 8 consecutive columns hit 32 distinct banks
constexpr int GS = 33;         // row stride of 32x32 Grams
constexpr int WS = 17;         // row stride of W
constexpr int RS = 72;         // row stride (elements) of the staged raw inputs: rows start 4 banks apart
constexpr float kTiny = 1e-20f;  // smallest cumulative decay the factorised form accepts
enum { VR = 0, VW = 1, VK = 2, VV = 3, VA = 4, VB = 5 };

// ---- bulk copies on the TMA engine (global -> shared), completed through
// an mbarrier's transaction count.
__device__ __forceinline__ unsigned smem_addr(const void *p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Bounded waits.  A wait polls for the completion of the mbarrier phase of
// this parity for at most kWaitLimitNs of the global timer (0.5 s; a chunk's
// copies land within microseconds).  The first wait of a CTA that runs out
// records the timeout in *err (read by wkv7_async_status) and sets the CTA's
// shared `lost` flag; from then on every wait of that CTA returns at once, the
// kernel leaves its chunk loop at the next chunk start and only a final drain
// (mbar_drain, also bounded) remains, so a lost copy costs a CTA at most two
// limits (about 1 s) instead of hanging the GPU.
constexpr unsigned long long kWaitLimitNs = 500ull * 1000ull * 1000ull;
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, unsigned *err, volatile int *lost) {
    if (mbar_test(bar, parity)) return true;
    if (*lost) return false;
    const unsigned long long t0 = global_ns();
    for (unsigned n = 1;; ++n) {
        if (mbar_test(bar, parity)) return true;
        if ((n & 31u) == 0) {
            if (*lost) return false;
            if (global_ns() - t0 > kWaitLimitNs) break;
        }
    }
    *lost = 1;
    if (err) atomicOr(err, 1u);
    return false;
}
// Before a CTA that lost a wait exits: wait (bounded as above) for the copies
// still addressed to this phase, so that none lands in shared memory the CTA
// no longer owns.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, unsigned parity) {
    const unsigned long long t0 = global_ns();
    for (unsigned n = 1; !mbar_test(bar, parity); ++n)
        if ((n & 31u) == 0 && global_ns() - t0 > kWaitLimitNs) return;
}
// Test-only builds (-DWKV7_TEST_PHANTOM_TX) announce kPhantomTx bytes more than
// one chunk's copies deliver, so that the wait for that chunk runs out without
// anything else going wrong.
#ifdef WKV7_TEST_PHANTOM_TX
constexpr unsigned kPhantomTx = 16;
#else
constexpr unsigned kPhantomTx = 0;
#endif
// One contiguous block, both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}
// Tensor copies of a chunk's input rows: 4-D maps over [B][T][H][64] (r, w,
// k, v, a, b and, for the backward, dy), box RS x 1 x C x 1, so that one copy
// fills a padded [C][RS] staging block; the columns past 64 and the tokens
// past T are out of range and arrive as zeros.
struct InputMaps {
    // r, w, k, v, a, b; then dy (backward) or y; then the checkpoints (forward); then the
    // epilogue's o (forward) or the forward's y (backward) of the GroupNorm + bonus calls
    CUtensorMap m[9];
};
__device__ __forceinline__ void tma_rows(void *dst, const CUtensorMap *map, int h, int t0, int b, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];\n" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(h), "r"(t0), "r"(b), "r"(smem_addr(bar))
        : "memory");
}

// Tensor stores of a chunk's gradient tiles: maps over [B][T][H][64] fp32 with
// box OS x 1 x C x 1 read from padded [C][OS] staging blocks (OS = 68 keeps
// the accumulator-layout writes into them free of bank conflicts); the
// columns past 64 and the tokens past T are out of range and not written.
constexpr int OS = 68;
struct OutputMaps {
    CUtensorMap m[6];
};
__device__ __forceinline__ void tma_store_rows(const CUtensorMap *map, const void *src, int h, int t0, int b) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_addr(src)), "r"(0), "r"(h), "r"(t0), "r"(b)
                 : "memory");
}
// 2-D tensor copy into shared memory: box at (column 0, row `row`).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int row, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_addr(bar))
        : "memory");
}
// Fetch the same box into L2 only (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int row) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(0), "r"(row)
                 : "memory");
}
// 2-D tensor store: box at (column 0, row `row`).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int row) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_addr(src)), "r"(0), "r"(row)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// The shared sources of this thread's committed bulk stores may be reused.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// This thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// Orders this thread's earlier generic-proxy shared accesses before later
// async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

template <typename E>
__device__ __forceinline__ float ld_raw(const E *raw, int vec, int t, int j);
template <>
__device__ __forceinline__ float ld_raw<float>(const float *raw, int vec, int t, int j) {
    return raw[(vec * C + t) * RS + j];
}
template <>
__device__ __forceinline__ float ld_raw<__nv_bfloat16>(const __nv_bfloat16 *raw, int vec, int t, int j) {
    return __bfloat162float(raw[(vec * C + t) * RS + j]);
}

// The recurrence's w, a and b at (t, j) from the staged rows.  With kP the
// staged w, a and b rows hold the producers' inputs ("timemix.cu" page,
// k_decay and k_composites): w = exp(-0.606531 sigmoid(w_pre)), a = -kk,
// b = kk * avec.
// The hardware exponential and reciprocal (__expf, __fdividef: a few ulp,
// about 3e-7 relative here, far below the split-bf16 product error) keep
// these off the per-chunk decay chain's critical path; the forward and the
// backward evaluate the same expressions, so both see the same decays.
constexpr float kDecayScale = 0.606531f;
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
template <bool kP, typename E>
__device__ __forceinline__ float in_w(const E *raw, int t, int j) {
    const float x = ld_raw(raw, VW, t, j);
    return kP ? __expf(-kDecayScale * sigmoid_f(x)) : x;
}
template <bool kP, typename E>
__device__ __forceinline__ float in_a(const E *raw, int t, int j) {
    const float x = ld_raw(raw, VA, t, j);
    return kP ? -x : x;
}
template <bool kP, typename E>
__device__ __forceinline__ float in_b(const E *raw, int t, int j) {
    return kP ? ld_raw(raw, VA, t, j) * ld_raw(raw, VB, t, j) : ld_raw(raw, VB, t, j);
}

// Elements j .. j + 3 (j % 4 == 0) of a staged row as one 64/128-bit load.
template <typename E>
__device__ __forceinline__ float4 ld_raw4(const E *raw, int vec, int t, int j);
template <>
__device__ __forceinline__ float4 ld_raw4<float>(const float *raw, int vec, int t, int j) {
    return *reinterpret_cast<const float4 *>(raw + (vec * C + t) * RS + j);
}
template <>
__device__ __forceinline__ float4 ld_raw4<__nv_bfloat16>(const __nv_bfloat16 *raw, int vec, int t, int j) {
    const uint2 u = *reinterpret_cast<const uint2 *>(raw + (vec * C + t) * RS + j);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}

template <typename E>
__host__ __device__ constexpr size_t raw_bytes() { return (size_t)6 * C * RS * sizeof(E); }

// Host: the driver's tensor-map encoder, looked up through the runtime so
// that the library does not link against the driver library itself.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn encode_tiled_fn() {
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Host: encode the row map of one [B][T][H][64] tensor (element size esize),
// box width `box0` elements (RS for the input staging, OS for gradient tiles).
inline cudaError_t encode_rows_map(CUtensorMap *m, const void *base, int esize, int B, int T, int H, int box0 = RS) {
    const EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[4] = {64, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {64ull * esize, 64ull * esize * H, 64ull * esize * H * T};
    const cuuint32_t box[4] = {(cuuint32_t)box0, 1, C, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = encode(
        m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(base),
        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
// Host: maps of the six inputs, and of dy when given.
inline cudaError_t encode_input_maps(InputMaps *maps, const SeqArgs &p, const float *dy) {
    const int es = p.dtype == 1 ? 2 : 4;
    const void *src[6] = {p.r, p.w, p.k, p.v, p.a, p.b};
    for (int i = 0; i < 6; ++i) {
        const cudaError_t e = encode_rows_map(&maps->m[i], src[i], es, p.B, p.T, p.H);
        if (e != cudaSuccess) return e;
    }
    return dy ? encode_rows_map(&maps->m[6], dy, 4, p.B, p.T, p.H) : cudaSuccess;
}
// Host: map of the checkpoints as rows of 64 fp32 (nrows = B*H*ceil(T/L)*64),
// box box_cols x box_rows (padded staging rows, the columns past 64 clipped on
// stores and zero-filled on loads: eight state rows of one warp for the
// stores, a whole 64-row state for the loads).
inline cudaError_t encode_ckpt_map(CUtensorMap *m, const float *ckpt, long long nrows, int box_rows = 8,
                                   int box_cols = OS) {
    const EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {64, (cuuint64_t)nrows};
    const cuuint64_t strides[1] = {64ull * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ckpt), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
// Host: maps of the six gradients dr, dw, dk, dv, da, db (fp32).
inline cudaError_t encode_output_maps(OutputMaps *maps, const SeqArgs &p) {
    float *const dst[6] = {p.dr, p.dw, p.dk, p.dv, p.da, p.db};
    for (int i = 0; i < 6; ++i) {
        const cudaError_t e = encode_rows_map(&maps->m[i], dst[i], 4, p.B, p.T, p.H, OS);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Sum over the 32 lanes of a warp, returned to every lane.
__device__ __forceinline__ float warp_allsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// The GroupNorm epsilon of the output epilogue ("timemix.cu" page, k_groupnorm).
constexpr float kGnEps = 64e-5f;

// Hardware approximate reciprocal (rcp.approx, about 1 ulp); used for 1/d_t,
// whose rounding is far below the split-bf16 product error.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float4 mul4(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
// a and b at (t, j .. j + 3), as in_a / in_b
template <bool kP, typename E>
__device__ __forceinline__ float4 in_a4(const E *raw, int t, int j) {
    const float4 x = ld_raw4(raw, VA, t, j);
    return kP ? make_float4(-x.x, -x.y, -x.z, -x.w) : x;
}
template <bool kP, typename E>
__device__ __forceinline__ float4 in_b4(const E *raw, int t, int j) {
    return kP ? mul4(ld_raw4(raw, VA, t, j), ld_raw4(raw, VB, t, j)) : ld_raw4(raw, VB, t, j);
}
__device__ __forceinline__ float4 rcp4(float4 a) {
    return make_float4(rcp_approx(a.x), rcp_approx(a.y), rcp_approx(a.z), rcp_approx(a.w));
}

// d_t per key column (threads first_thread .. first_thread + 63; with the
// fused producers all 128 threads, two per key); padding tokens (t >= nv)
// decay by 1.
// Returns true (on the calling thread) when some d_t of its column leaves
// [1e-20, 1e20] (or is not finite): the factorised form then cannot divide
// by d_t and the chunk takes the exact per-token path.  With kMinW (the
// plain backward) a decay w_t below kSmallW also sends the chunk there: the
// backward recovers dw_t from the running sum of w_t o dw_t by a division by
// w_t, which multiplies that sum's absolute rounding (about 1e-5 of the
// largest r o dr term) by 1 / w_t.
constexpr float kSmallW = 0.0625f;
// With kP, sig (if not NULL) receives sigmoid(w_pre) of every staged token,
// [t][j] with row stride DS, for callers that need it again.
template <bool kP, typename E, bool kMinW = false>
__device__ __forceinline__ bool prep_decay(const E *raw, float *dd, int nv, int first_thread = 0,
                                           float *sig = nullptr) {
    bool bad = false;
    if constexpr (kP) {
        // the producers' exponentials on all four warps: warp w holds keys
        // 16w..16w+15, lanes 0-15 tokens 0..7 and lanes 16-31 tokens 8..15 of key
        // 16w + lane % 16; the second half continues from the first half's
        // product with one shuffle (first_thread is not used)
        const int lane = threadIdx.x & 31, j = 16 * (threadIdx.x >> 5) + (lane & 15), t0 = 8 * (lane >> 4);
        float wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // in_w<true>, with the sigmoid kept
            const float sg = sigmoid_f(ld_raw(raw, VW, t0 + u, j));
            if (sig) sig[(t0 + u) * DS + j] = sg;
            wv[u] = t0 + u < nv ? __expf(-kDecayScale * sg) : 1.f;
        }
        float dl[8], dc = 1.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            dc = __fmul_rn(dc, wv[u]);
            dl[u] = dc;
        }
        const float head = __shfl_sync(0xffffffffu, dc, lane & 15);  // d_7 of the key
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float d = lane >= 16 ? __fmul_rn(dl[u], head) : dl[u];
            dd[(t0 + u) * DS + j] = d;
            bad |= !(d >= kTiny && d <= 1.f / kTiny);
        }
        return bad;
    }
    const int j = (int)threadIdx.x - first_thread;
    if (j >= 0 && j < 64) {
        // all loads first: the product chain then runs at FMUL latency
        float wv[C];
#pragma unroll
        for (int t = 0; t < C; ++t) wv[t] = t < nv ? in_w<kP>(raw, t, j) : 1.f;
        float dc = 1.f;
#pragma unroll
        for (int t = 0; t < C; ++t) {
            dc = __fmul_rn(dc, wv[t]);
            dd[t * DS + j] = dc;
            bad |= !(dc >= kTiny && dc <= 1.f / kTiny);
            if constexpr (kMinW) bad |= !(wv[t] >= kSmallW);
        }
    }
    return bad;
}

// W = (I - M_b)^{-1} (unit upper triangular) by back substitution: lanes
// 0..15 of warp 0 each build one column.
__device__ __forceinline__ void prep_inverse(const float *G, float *Wm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp != 0 || lane >= C) return;
    const int t = lane;
    float wc[C];
#pragma unroll
    for (int s = C - 1; s >= 0; --s) {
        // sum the terms of the rows found longest ago first, so that only one
        // FMA depends on the row computed just before (wc[s + 1])
        float acc = (s == t) ? 1.f : 0.f;
#pragma unroll
        for (int u = C - 1; u > s; --u) acc = __fmaf_rn(G[s * GS + u], wc[u], acc);
        wc[s] = acc;
    }
#pragma unroll
    for (int s = 0; s < C; ++s) Wm[s * WS + t] = wc[s];
}

// W = (I - M_b)^{-1} as above, M_b read from a row-major copy with row
// stride MBS floats (16-byte aligned rows, unpadded: every lane reads the
// same row, a broadcast): each row comes in with broadcast
// 16-byte loads issued ahead of the product chain.  Lane t holds column t of
// W and writes it, split into bf16 hi + lo, as row t of W^T in two compact
// 16 x 16 matrices of row stride CS (four 16-byte stores per lane).
constexpr int MBS = 16;
constexpr int CS = 24;  // row stride (elements) of a compact 16 x 16 split matrix: ldmatrix rows 12 banks apart
__device__ __forceinline__ void prep_inverse_t(const float *Mb, __nv_bfloat16 *wt_hi, __nv_bfloat16 *wt_lo) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp != 0 || lane >= C) return;
    const int t = lane;
    float wc[C];
#pragma unroll
    for (int s = C - 1; s >= 0; --s) {
        const float4 *r4 = reinterpret_cast<const float4 *>(Mb + s * MBS);
        float m[C];
#pragma unroll
        for (int k = (s + 1) >> 2; k < 4; ++k) {
            const float4 x = r4[k];
            m[4 * k] = x.x; m[4 * k + 1] = x.y; m[4 * k + 2] = x.z; m[4 * k + 3] = x.w;
        }
        float acc = (s == t) ? 1.f : 0.f;
#pragma unroll
        for (int u = C - 1; u > s; --u) acc = __fmaf_rn(m[u], wc[u], acc);
        wc[s] = acc;
    }
    uint32_t h[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const Frag2 f = split2(wc[2 * i], wc[2 * i + 1]);
        h[i] = f.hi;
        l[i] = f.lo;
    }
    uint4 *hp = reinterpret_cast<uint4 *>(wt_hi + t * CS), *lp = reinterpret_cast<uint4 *>(wt_lo + t * CS);
    hp[0] = make_uint4(h[0], h[1], h[2], h[3]);
    hp[1] = make_uint4(h[4], h[5], h[6], h[7]);
    lp[0] = make_uint4(l[0], l[1], l[2], l[3]);
    lp[1] = make_uint4(l[4], l[5], l[6], l[7]);
}

}  // namespace chunk
}  // namespace wkv7
