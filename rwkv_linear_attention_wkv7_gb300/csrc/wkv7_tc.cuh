// Fifth-generation tensor-core (tcgen05) helpers for the chunked WKV7 kernels:
// the canonical no-swizzle operand layout in shared memory, shared-memory
// matrix descriptors, the instruction descriptor of a bf16 x bf16 -> fp32 MMA,
// the single-thread MMA issue with completion on an mbarrier, and the
// tensor-memory (TMEM) allocation and loads.
//
// Canonical layout (no swizzle).  A matrix of R rows x NC columns of bf16
// (NC % 8 == 0) is stored as 8 x 8 "core matrices" of 128 contiguous bytes
// (8 rows of 16 bytes); core (rg, cg) starts at byte rg * 16 NC + cg * 128.
// The same bytes serve both operand majors of tcgen05.mma:
//   rows = M (or N), columns = K ("K-major"):  LBO = 128 (next 8 columns of K),
//                                              SBO = 16 NC (next 8 rows of M);
//   rows = K, columns = M (or N) ("MN-major"): LBO = 16 NC (next 8 rows of K),
//                                              SBO = 128 (next 8 columns of M).
// One MMA of kind::f16 consumes K = 16, so successive K steps start 256 bytes
// (K-major) or 32 NC bytes (MN-major) further on.  Every 8-element row segment
// is 16 contiguous bytes, so ldmatrix / stmatrix address the same layout one
// core matrix per 8 x 8 tile (conflict-free).
//
// The accumulator of an M = 64 MMA (cta_group::1) holds row 16 w + r in TMEM
// lane 32 w + r (r < 16) and column n in TMEM column n; a tcgen05.ld of shape
// 16x256b by warp w returns, per 8 columns, exactly the fp32 accumulator
// fragment of mma.sync.m16n8 (rows g, g + 8; columns 2 q, 2 q + 1).  Both
// facts, and the descriptor field meanings below, were checked on the GB300
// by a probe of every layout against a host reference.
#pragma once
#include <stdint.h>

#include "wkv7_mma.cuh"

namespace wkv7 {
namespace tc {

// element offset of (r, c) in a canonical matrix of NC columns
template <int NC>
__device__ __forceinline__ int cof(int r, int c) {
    return ((r >> 3) * NC + (c & ~7)) * 8 + (r & 7) * 8 + (c & 7);
}

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Shared-memory matrix descriptor: start address >> 4 in bits [0,14), LBO >> 4
// in [16,30), SBO >> 4 in [32,46), descriptor version 1 in [46,48), no swizzle
// (layout type 0 in [61,64)).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}
// Descriptor of K step ks of a canonical matrix of NC columns whose hi or lo
// part starts at `addr`: K-major (columns = K) or MN-major (rows = K).
template <int NC>
__device__ __forceinline__ uint64_t kdesc(uint32_t addr, int ks) {
    return sdesc(addr + ks * 256, 128, 16 * NC);
}
template <int NC>
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, int ks) {
    return sdesc(addr + ks * 32 * NC, 16 * NC, 128);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits [4,6) = 1), A and
// B bf16 (bits [7,10) = [10,13) = 1), A / B major (bit 15 / 16: 1 = MN-major),
// N >> 3 in bits [17,23), M >> 4 in bits [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A B^T, A and B read from shared memory through descriptors;
// `acc` = false overwrites D.  Issued by one thread.
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc)
        : "memory");
}
// A split product over one K step: D (+)= A_lo B_hi + A_hi B_lo + A_hi B_hi
// (the three products of the bf16x3 scheme of wkv7_mma.cuh).
__device__ __forceinline__ void mma3(uint32_t d, uint64_t a_hi, uint64_t a_lo, uint64_t b_hi, uint64_t b_lo,
                                     uint32_t id, bool acc) {
    mma(d, a_lo, b_hi, id, acc);
    mma(d, a_hi, b_lo, id, true);
    mma(d, a_hi, b_hi, id, true);
}
// The mbarrier receives one arrival once every MMA this thread issued before
// has completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM allocation by one whole warp; the column base is written to *slot.
__device__ __forceinline__ void alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

// 16 lanes x 32 columns of this warp's quarter (lane base 32 w) as four
// accumulator fragments: c[n][0..3] = (row g, cols 8n + 2q, +1), (row g + 8, ...).
__device__ __forceinline__ void ld32(uint32_t taddr, float c[4][4]) {
    uint32_t r[16];
    // load and wait in one statement: the registers are defined only once the load has completed
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[n][e] = __uint_as_float(r[4 * n + e]);
}
// TMEM address of column `col` in warp w's lane quarter.
__device__ __forceinline__ uint32_t taddr(uint32_t base, int warp, int col) {
    return base + ((uint32_t)(32 * warp) << 16) + (uint32_t)col;
}

// ---- canonical-layout versions of the ldmatrix / stmatrix operand helpers of
// wkv7_mma.cuh (same fragments, core-matrix addressing)
template <int NC>
__device__ __forceinline__ AFrag lda(const HL &M, int m0, int k0, int lane) {  // A[m][k] = M[m0 + m][k0 + k]
    const int off = cof<NC>(m0 + (lane & 7) + 8 * ((lane >> 3) & 1), k0 + 8 * (lane >> 4));
    AFrag f;
    ldsm_x4(f.hi, M.hi + off);
    ldsm_x4(f.lo, M.lo + off);
    return f;
}
template <int NC>
__device__ __forceinline__ AFrag lda_t(const HL &M, int m0, int k0, int lane) {  // A[m][k] = M[k0 + k][m0 + m]
    const int off = cof<NC>(k0 + (lane & 7) + 8 * (lane >> 4), m0 + 8 * ((lane >> 3) & 1));
    AFrag f;
    ldsm_x4_t(f.hi, M.hi + off);
    ldsm_x4_t(f.lo, M.lo + off);
    return f;
}
template <int NC>
__device__ __forceinline__ AFrag lda_hi(const HL &M, int m0, int k0, int lane) {  // lo part known to be zero
    const int off = cof<NC>(m0 + (lane & 7) + 8 * ((lane >> 3) & 1), k0 + 8 * (lane >> 4));
    AFrag f;
    ldsm_x4(f.hi, M.hi + off);
    f.lo[0] = f.lo[1] = f.lo[2] = f.lo[3] = 0u;
    return f;
}
// B fragments of n-tiles n0.., n0 + 8.., B[k][n] = M[n][k]
template <int NC>
__device__ __forceinline__ void ldb2(const HL &M, int n0, int k0, int lane, BFrag &b0, BFrag &b1) {
    const int off = cof<NC>(n0 + (lane & 7) + 8 * (lane >> 4), k0 + 8 * ((lane >> 3) & 1));
    uint32_t h[4], l[4];
    ldsm_x4(h, M.hi + off);
    ldsm_x4(l, M.lo + off);
    b0.hi[0] = h[0]; b0.hi[1] = h[1]; b1.hi[0] = h[2]; b1.hi[1] = h[3];
    b0.lo[0] = l[0]; b0.lo[1] = l[1]; b1.lo[0] = l[2]; b1.lo[1] = l[3];
}
// B fragments of n-tiles n0.., n0 + 8.., B[k][n] = M[k][n]
template <int NC>
__device__ __forceinline__ void ldb2_t(const HL &M, int n0, int k0, int lane, BFrag &b0, BFrag &b1) {
    const int off = cof<NC>(k0 + (lane & 7) + 8 * ((lane >> 3) & 1), n0 + 8 * (lane >> 4));
    uint32_t h[4], l[4];
    ldsm_x4_t(h, M.hi + off);
    ldsm_x4_t(l, M.lo + off);
    b0.hi[0] = h[0]; b0.hi[1] = h[1]; b1.hi[0] = h[2]; b1.hi[1] = h[3];
    b0.lo[0] = l[0]; b0.lo[1] = l[1]; b1.lo[0] = l[2]; b1.lo[1] = l[3];
}
// 16 x 16 accumulator block (two n-tiles) split and stored at M[row0 + m][col0 + n]
template <int NC>
__device__ __forceinline__ void st_acc16(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row0, int col0, const float c[2][4],
                                         int lane) {
    const Frag2 f0 = split2(c[0][0], c[0][1]), f1 = split2(c[0][2], c[0][3]);
    const Frag2 f2 = split2(c[1][0], c[1][1]), f3 = split2(c[1][2], c[1][3]);
    const int k = lane >> 3, r = lane & 7;
    const int off = cof<NC>(row0 + 8 * (k & 1) + r, col0 + 8 * (k >> 1));
    stsm_x4(hi + off, f0.hi, f1.hi, f2.hi, f3.hi);
    stsm_x4(lo + off, f0.lo, f1.lo, f2.lo, f3.lo);
}
// the same block stored transposed: M[row0 + n][col0 + m] = block[m][n]
template <int NC>
__device__ __forceinline__ void st_acc_t16(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row0, int col0,
                                           const float c[2][4], int lane) {
    const Frag2 f0 = split2(c[0][0], c[0][1]), f1 = split2(c[0][2], c[0][3]);
    const Frag2 f2 = split2(c[1][0], c[1][1]), f3 = split2(c[1][2], c[1][3]);
    const int k = lane >> 3, r = lane & 7;
    const int off = cof<NC>(row0 + 8 * (k >> 1) + r, col0 + 8 * (k & 1));
    stsm_x4_t(hi + off, f0.hi, f1.hi, f2.hi, f3.hi);
    stsm_x4_t(lo + off, f0.lo, f1.lo, f2.lo, f3.lo);
}
// split of four consecutive values at M[row][col .. col + 3] (col % 4 == 0)
template <int NC>
__device__ __forceinline__ void st_hl4(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row, int col, float4 x) {
    const Frag2 f0 = split2(x.x, x.y), f1 = split2(x.z, x.w);
    const int off = cof<NC>(row, col);
    *reinterpret_cast<uint2 *>(hi + off) = make_uint2(f0.hi, f1.hi);
    *reinterpret_cast<uint2 *>(lo + off) = make_uint2(f0.lo, f1.lo);
}
// split of eight consecutive values at M[row][col .. col + 7] (col % 8 == 0): one 16-byte store per part
template <int NC>
__device__ __forceinline__ void st_hl8(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row, int col, float4 x, float4 y) {
    const Frag2 f0 = split2(x.x, x.y), f1 = split2(x.z, x.w), f2 = split2(y.x, y.y), f3 = split2(y.z, y.w);
    const int off = cof<NC>(row, col);
    *reinterpret_cast<uint4 *>(hi + off) = make_uint4(f0.hi, f1.hi, f2.hi, f3.hi);
    *reinterpret_cast<uint4 *>(lo + off) = make_uint4(f0.lo, f1.lo, f2.lo, f3.lo);
}
// (hi + lo) of M[row][col], M[row][col + 1] (col even)
template <int NC>
__device__ __forceinline__ float2 ld_hl(const HL &M, int row, int col) {
    const int off = cof<NC>(row, col);
    const uint32_t h = *reinterpret_cast<const uint32_t *>(M.hi + off);
    const uint32_t l = *reinterpret_cast<const uint32_t *>(M.lo + off);
    return make_float2(__uint_as_float(h << 16) + __uint_as_float(l << 16),
                       __uint_as_float(h & 0xffff0000u) + __uint_as_float(l & 0xffff0000u));
}

}  // namespace tc
}  // namespace wkv7
