// Warp-level tensor-core helpers for the chunked WKV7 kernels: bf16 m16n8k16
// MMA with fp32 accumulation, and the three-product split ("bf16x3") that
// recovers about 17 bits of operand precision: x = hi + lo with hi = bf16(x),
// lo = bf16(x - hi); a*b ~ hi_a*hi_b + hi_a*lo_b + lo_a*hi_b.
//
// Fragment layouts (PTX ISA, mma.m16n8k16 with .bf16): lane l, g = l/4,
// q = l%4.  A (16x16, row major): a0 = A[g][2q..2q+1], a1 = A[g+8][2q..],
// a2 = A[g][2q+8..], a3 = A[g+8][2q+8..].  B (16x8): b0 = B[2q..2q+1][g],
// b1 = B[2q+8..2q+9][g].  C (16x8, fp32): c0,c1 = C[g][2q..2q+1],
// c2,c3 = C[g+8][2q..2q+1].  The lower half of each 32-bit register holds the
// element with the smaller k index.
#pragma once
#include <stdint.h>
#include <cuda_bf16.h>

namespace wkv7 {

struct Frag2 {  // one 32-bit bf16x2 register as hi and lo parts
    uint32_t hi, lo;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float x0, float x1) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x1), "f"(x0));
    return r;
}

// Split (x0, x1) into bf16x2 hi and lo registers.
__device__ __forceinline__ Frag2 split2(float x0, float x1) {
    Frag2 f;
    f.hi = pack_bf16x2(x0, x1);
    const float h0 = __uint_as_float(f.hi << 16);
    const float h1 = __uint_as_float(f.hi & 0xffff0000u);
    f.lo = pack_bf16x2(x0 - h0, x1 - h1);
    return f;
}

// Pure register operation: not volatile, so the compiler may interleave
// independent accumulators (the three products of one split MMA are serial).
__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], const uint32_t b[2]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// A operand (16x16) split into hi and lo fragments.
struct AFrag {
    uint32_t hi[4], lo[4];
};
// B operand (16x8) split into hi and lo fragments.
struct BFrag {
    uint32_t hi[2], lo[2];
};

// c += A*B with split operands: small cross terms first, then hi*hi.
__device__ __forceinline__ void mma3(float c[4], const AFrag &a, const BFrag &b) {
    mma_bf16(c, a.lo, b.hi);
    mma_bf16(c, a.hi, b.lo);
    mma_bf16(c, a.hi, b.hi);
}

// A fragment from four fp32 pairs: (r0: row g, k 2q..), (r1: row g+8, k 2q..),
// (r2: row g, k 2q+8..), (r3: row g+8, k 2q+8..).
__device__ __forceinline__ AFrag make_a(float2 r0, float2 r1, float2 r2, float2 r3) {
    AFrag f;
    Frag2 t;
    t = split2(r0.x, r0.y); f.hi[0] = t.hi; f.lo[0] = t.lo;
    t = split2(r1.x, r1.y); f.hi[1] = t.hi; f.lo[1] = t.lo;
    t = split2(r2.x, r2.y); f.hi[2] = t.hi; f.lo[2] = t.lo;
    t = split2(r3.x, r3.y); f.hi[3] = t.hi; f.lo[3] = t.lo;
    return f;
}
__device__ __forceinline__ BFrag make_b(float2 k0, float2 k8) {
    BFrag f;
    Frag2 t;
    t = split2(k0.x, k0.y); f.hi[0] = t.hi; f.lo[0] = t.lo;
    t = split2(k8.x, k8.y); f.hi[1] = t.hi; f.lo[1] = t.lo;
    return f;
}

// fp32 values of an A fragment's 8 elements (hi + lo), in C-tile order:
// v[0..1] = (row g, k 2q..2q+1), v[2..3] = (row g+8, ..), v[4..5] = (row g, k 2q+8..), v[6..7] = (row g+8, ..)
__device__ __forceinline__ void a_values(const AFrag &f, float v[8]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        v[2 * r] = __uint_as_float(f.hi[r] << 16) + __uint_as_float(f.lo[r] << 16);
        v[2 * r + 1] = __uint_as_float(f.hi[r] & 0xffff0000u) + __uint_as_float(f.lo[r] & 0xffff0000u);
    }
}

// A fragment for k-tile kt from a 16-row x 64-column fp32 accumulator slab
// held as 8 n-tiles of C fragments (c[nt][0..3]): the C layout of n-tiles
// 2kt and 2kt+1 is exactly the A layout of k-tile kt.
__device__ __forceinline__ AFrag a_from_acc(const float c[][4], int kt) {
    return make_a(make_float2(c[2 * kt][0], c[2 * kt][1]), make_float2(c[2 * kt][2], c[2 * kt][3]),
                  make_float2(c[2 * kt + 1][0], c[2 * kt + 1][1]), make_float2(c[2 * kt + 1][2], c[2 * kt + 1][3]));
}

}  // namespace wkv7

namespace wkv7 {

// ---- bf16 hi/lo operand matrices in shared memory, loaded with ldmatrix.
// A matrix is stored twice (hi and lo parts), row-major, row stride MS
// elements (144 bytes: the eight rows of an 8x8 ldmatrix tile start in
// distinct bank groups).
constexpr int MS = 72;

__device__ __forceinline__ void ldsm_x4(uint32_t r[4], const void *p) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], const void *p) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

struct HL {  // a split operand matrix: hi and lo parts, same layout
    const __nv_bfloat16 *hi, *lo;
};

// A fragment, A[m][k] = M[m0 + m][k0 + k] (M stored [m][k], row stride S).
template <int S = MS>
__device__ __forceinline__ AFrag lda(const HL &M, int m0, int k0, int lane) {
    const int off = (m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * S + k0 + 8 * (lane >> 4);
    AFrag f;
    ldsm_x4(f.hi, M.hi + off);
    ldsm_x4(f.lo, M.lo + off);
    return f;
}
// A fragment, A[m][k] = M[k0 + k][m0 + m] (M stored [k][m], row stride S).
template <int S = MS>
__device__ __forceinline__ AFrag lda_t(const HL &M, int m0, int k0, int lane) {
    const int off = (k0 + (lane & 7) + 8 * (lane >> 4)) * S + m0 + 8 * ((lane >> 3) & 1);
    AFrag f;
    ldsm_x4_t(f.hi, M.hi + off);
    ldsm_x4_t(f.lo, M.lo + off);
    return f;
}
// B fragments of two n-tiles (n0..n0+7, n0+8..n0+15), B[k][n] = M[n][k] (M stored [n][k],
// row stride S).
template <int S = MS>
__device__ __forceinline__ void ldb2(const HL &M, int n0, int k0, int lane, BFrag &b0, BFrag &b1) {
    const int off = (n0 + (lane & 7) + 8 * (lane >> 4)) * S + k0 + 8 * ((lane >> 3) & 1);
    uint32_t h[4], l[4];
    ldsm_x4(h, M.hi + off);
    ldsm_x4(l, M.lo + off);
    b0.hi[0] = h[0]; b0.hi[1] = h[1]; b1.hi[0] = h[2]; b1.hi[1] = h[3];
    b0.lo[0] = l[0]; b0.lo[1] = l[1]; b1.lo[0] = l[2]; b1.lo[1] = l[3];
}
// The same two B fragments with hi only (lo set to zero), for a matrix whose
// lo part is identically zero.
__device__ __forceinline__ void ldb2_hi(const HL &M, int n0, int k0, int lane, BFrag &b0, BFrag &b1) {
    const int off = (n0 + (lane & 7) + 8 * (lane >> 4)) * MS + k0 + 8 * ((lane >> 3) & 1);
    uint32_t h[4];
    ldsm_x4(h, M.hi + off);
    b0.hi[0] = h[0]; b0.hi[1] = h[1]; b1.hi[0] = h[2]; b1.hi[1] = h[3];
    b0.lo[0] = b0.lo[1] = b1.lo[0] = b1.lo[1] = 0u;
}
// A fragment with hi only (lo set to zero), A[m][k] = M[m0 + m][k0 + k].
__device__ __forceinline__ AFrag lda_hi(const HL &M, int m0, int k0, int lane) {
    const int off = (m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * MS + k0 + 8 * (lane >> 4);
    AFrag f;
    ldsm_x4(f.hi, M.hi + off);
    f.lo[0] = f.lo[1] = f.lo[2] = f.lo[3] = 0u;
    return f;
}
// A fragment with hi only (lo set to zero), A[m][k] = M[k0 + k][m0 + m].
__device__ __forceinline__ AFrag lda_t_hi(const HL &M, int m0, int k0, int lane) {
    const int off = (k0 + (lane & 7) + 8 * (lane >> 4)) * MS + m0 + 8 * ((lane >> 3) & 1);
    AFrag f;
    ldsm_x4_t(f.hi, M.hi + off);
    f.lo[0] = f.lo[1] = f.lo[2] = f.lo[3] = 0u;
    return f;
}
// B fragments of two n-tiles, B[k][n] = M[k][n] (M stored [k][n], row stride S).
template <int S = MS>
__device__ __forceinline__ void ldb2_t(const HL &M, int n0, int k0, int lane, BFrag &b0, BFrag &b1) {
    const int off = (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * S + n0 + 8 * (lane >> 4);
    uint32_t h[4], l[4];
    ldsm_x4_t(h, M.hi + off);
    ldsm_x4_t(l, M.lo + off);
    b0.hi[0] = h[0]; b0.hi[1] = h[1]; b1.hi[0] = h[2]; b1.hi[1] = h[3];
    b0.lo[0] = l[0]; b0.lo[1] = l[1]; b1.lo[0] = l[2]; b1.lo[1] = l[3];
}
// Store the split of (x0, x1) at M[row][col], M[row][col + 1] (col even).
__device__ __forceinline__ void st_hl(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row, int col, float x0, float x1) {
    const Frag2 f = split2(x0, x1);
    *reinterpret_cast<uint32_t *>(hi + row * MS + col) = f.hi;
    *reinterpret_cast<uint32_t *>(lo + row * MS + col) = f.lo;
}
// Store the split of four consecutive values at M[row][col..col + 3] (col % 4 == 0).
__device__ __forceinline__ void st_hl4(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row, int col, float4 x) {
    const Frag2 f0 = split2(x.x, x.y), f1 = split2(x.z, x.w);
    *reinterpret_cast<uint2 *>(hi + row * MS + col) = make_uint2(f0.hi, f1.hi);
    *reinterpret_cast<uint2 *>(lo + row * MS + col) = make_uint2(f0.lo, f1.lo);
}
template <int S = MS>
__device__ __forceinline__ float2 ld_hl(const __nv_bfloat16 *hi, const __nv_bfloat16 *lo, int row, int col) {
    const uint32_t h = *reinterpret_cast<const uint32_t *>(hi + row * S + col);
    const uint32_t l = *reinterpret_cast<const uint32_t *>(lo + row * S + col);
    return make_float2(__uint_as_float(h << 16) + __uint_as_float(l << 16),
                       __uint_as_float(h & 0xffff0000u) + __uint_as_float(l & 0xffff0000u));
}

// ---- fragments to and from memory, 32 bytes per lane stored as two 16-byte
// halves 512 bytes apart (half h of lane l at uint4 index 32 h + l), so that
// every warp-wide 16-byte access covers 512 contiguous bytes.
// A fragment: {hi[0..3]}, {lo[0..3]}.
__device__ __forceinline__ void st_afrag(float *dst, const AFrag &f, int lane) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[lane] = make_uint4(f.hi[0], f.hi[1], f.hi[2], f.hi[3]);
    d[32 + lane] = make_uint4(f.lo[0], f.lo[1], f.lo[2], f.lo[3]);
}
__device__ __forceinline__ AFrag ld_afrag(const float *src, int lane) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    const uint4 h = s[lane], l = s[32 + lane];
    AFrag f;
    f.hi[0] = h.x; f.hi[1] = h.y; f.hi[2] = h.z; f.hi[3] = h.w;
    f.lo[0] = l.x; f.lo[1] = l.y; f.lo[2] = l.z; f.lo[3] = l.w;
    return f;
}
// The B fragments of the two 8-column n-tiles of X (16 x 16, B[k][n] = X[n][k])
// from X's two accumulator tiles c[kt] (rows = n, columns = 8kt + ...): the
// accumulator layout of X is the B layout of its transpose.  Stored as
// {b0.hi, b0.lo}, {b1.hi, b1.lo}.
__device__ __forceinline__ void st_bfrags_acc(float *dst, const float c[2][4], int lane) {
    const Frag2 a = split2(c[0][0], c[0][1]), b = split2(c[1][0], c[1][1]);
    const Frag2 e = split2(c[0][2], c[0][3]), f = split2(c[1][2], c[1][3]);
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    d[lane] = make_uint4(a.hi, b.hi, a.lo, b.lo);
    d[32 + lane] = make_uint4(e.hi, f.hi, e.lo, f.lo);
}
__device__ __forceinline__ void ld_bfrags(const float *src, int lane, BFrag &b0, BFrag &b1) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    const uint4 x = s[lane], y = s[32 + lane];
    b0.hi[0] = x.x; b0.hi[1] = x.y; b0.lo[0] = x.z; b0.lo[1] = x.w;
    b1.hi[0] = y.x; b1.hi[1] = y.y; b1.lo[0] = y.z; b1.lo[1] = y.w;
}
// Two fp32 accumulator tiles (8 values per lane) of one warp, same halves.
__device__ __forceinline__ void st_acc2(float *dst, const float c0[4], const float c1[4], int lane) {
    float4 *d = reinterpret_cast<float4 *>(dst);
    d[lane] = make_float4(c0[0], c0[1], c0[2], c0[3]);
    d[32 + lane] = make_float4(c1[0], c1[1], c1[2], c1[3]);
}
__device__ __forceinline__ void ld_acc2(const float *src, float c0[4], float c1[4], int lane) {
    const float4 *s = reinterpret_cast<const float4 *>(src);
    const float4 x = s[lane], y = s[32 + lane];
    c0[0] = x.x; c0[1] = x.y; c0[2] = x.z; c0[3] = x.w;
    c1[0] = y.x; c1[1] = y.y; c1[2] = y.z; c1[3] = y.w;
}

// c[n] += A B[n] for NB accumulators, the three split products of each
// interleaved across the accumulators so that no two consecutive MMAs
// depend on each other.
// kALo / kBLo = false drops the product of an operand whose lo part is
// identically zero (an input that is exact in bf16): it would add exact zeros.
template <int NB, bool kALo = true, bool kBLo = true>
__device__ __forceinline__ void mma3n(float (*c)[4], const AFrag &a, const BFrag *b) {
    if constexpr (kALo) {
#pragma unroll
        for (int n = 0; n < NB; ++n) mma_bf16(c[n], a.lo, b[n].hi);
    }
    if constexpr (kBLo) {
#pragma unroll
        for (int n = 0; n < NB; ++n) mma_bf16(c[n], a.hi, b[n].lo);
    }
#pragma unroll
    for (int n = 0; n < NB; ++n) mma_bf16(c[n], a.hi, b[n].hi);
}

// ---- transposed stores of accumulator blocks with stmatrix (.trans): the
// 16 x 16 fp32 block held as two n-tiles c[0], c[1] (rows g, g + 8; columns
// 8u + 2q, +1) is split and written as M[row0 + n][col0 + m] = block[m][n]
// into a hi/lo matrix pair with row stride MS.  Lane l gives the address of
// row l % 8 of 8x8 tile l / 8 (tiles: rows 0-7 / 8-15 of the block times
// columns 0-7 / 8-15, in the order of the fragment registers).
__device__ __forceinline__ void stsm_x4_t(void *p, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}
__device__ __forceinline__ void st_acc_t16(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row0, int col0, const float c[2][4],
                                           int lane) {
    const Frag2 f0 = split2(c[0][0], c[0][1]), f1 = split2(c[0][2], c[0][3]);
    const Frag2 f2 = split2(c[1][0], c[1][1]), f3 = split2(c[1][2], c[1][3]);
    const int k = lane >> 3, r = lane & 7;
    const int off = (row0 + 8 * (k >> 1) + r) * MS + col0 + 8 * (k & 1);
    stsm_x4_t(hi + off, f0.hi, f1.hi, f2.hi, f3.hi);
    stsm_x4_t(lo + off, f0.lo, f1.lo, f2.lo, f3.lo);
}

// Same block stored untransposed: M[row0 + m][col0 + n] = block[m][n].
__device__ __forceinline__ void stsm_x4(void *p, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(r0), "r"(r1), "r"(r2),
                 "r"(r3)
                 : "memory");
}
template <int S = MS>
__device__ __forceinline__ void st_acc16(__nv_bfloat16 *hi, __nv_bfloat16 *lo, int row0, int col0, const float c[2][4],
                                         int lane) {
    const Frag2 f0 = split2(c[0][0], c[0][1]), f1 = split2(c[0][2], c[0][3]);
    const Frag2 f2 = split2(c[1][0], c[1][1]), f3 = split2(c[1][2], c[1][3]);
    const int k = lane >> 3, r = lane & 7;
    const int off = (row0 + 8 * (k & 1) + r) * S + col0 + 8 * (k >> 1);
    stsm_x4(hi + off, f0.hi, f1.hi, f2.hi, f3.hi);
    stsm_x4(lo + off, f0.lo, f1.lo, f2.lo, f3.lo);
}

}  // namespace wkv7
