// Floored remainder by a per-head invariant divisor, for the PLE row-id hash.
//
// The hash ends every head with floormod(mix, vocab) where floormod follows
// torch.remainder: the result takes the divisor's sign (FreeToken PR #338,
// "perf(ple): fuse the n-gram row-id hash into one Triton kernel", section
// "Why it is safe": the kernel fixes the sign of a truncated remainder).
//
// A generic 64-bit % is a long software routine on the GPU and would make the
// hash ALU-bound, so each divisor is turned once per thread block into a
// reciprocal and every remainder then costs a few multiplies:
//
//   Barrett reduction (P. Barrett, "Implementing the Rivest Shamir and
//   Adleman public key encryption algorithm on a standard digital signal
//   processor", CRYPTO 1986; the invariant-divisor form of T. Granlund and
//   P. Montgomery, "Division by invariant integers using multiplication",
//   PLDI 1994).  With d >= 1 and m = floor((2^64 - 1) / d), for any a < 2^64
//   the estimate q' = floor(a * m / 2^64) satisfies q - 1 <= q' <= q, where
//   q = floor(a / d):  m >= 2^64/d - 1 gives a*m/2^64 > a/d - 1, and
//   m <= (2^64-1)/d gives a*m/2^64 < a/d.  So r' = a - q'*d lies in [0, 2d).
//
//   When d <= 2^29, every remainder estimate below fits 32 bits, so only the
//   low 32 bits of q' are needed: bits 64..95 of the 128-bit product a*m.
//
// The sign without a branch on it: the signed mix x is read in offset binary,
// u = x + 2^63 (flip the top bit), so u is an unsigned value in [0, 2^64) and
//   floormod(x, d) = (u - 2^63) mod d = (u mod d + d - (2^63 mod d)) mod d.
// With D = d - (2^63 mod d) in [1, d] precomputed per head, adding D and a
// few conditional subtractions finish the floored remainder; each is
// min(r, r - k) on unsigned values (r - k wraps above r when r < k).
// A negative divisor follows from floormod(x, v) = r ? r - |v| : 0 with
// r = floormod(x, |v|), since the floored result lies in (v, 0].
#pragma once

#include <stdint.h>

namespace ple {

enum : uint32_t {
    kHeadNegative = 1u,  // vocab < 0
    kHeadZero = 2u,      // vocab == 0: the row is the offset
    kHeadFast = 4u,      // 0 < vocab <= 2^29: 32-bit remainder path
};

// One head's constants, kept structure-of-arrays in shared memory so the
// fast path reads 16 bytes per head and the offset separately:
//   fast  = {m_lo, m_hi, -2|v| mod 2^32 (fast heads), D low word},
//           m = floor((2^64-1)/|v|), D = |v| - (2^63 mod |v|)
//   off   = the head's row offset
//   ext   = {|v| high word, D high word, kHead* flags, |v| low word}
struct HeadConst {
    uint4 fast;
    int64_t off;
    uint4 ext;
};

__host__ __device__ __forceinline__ HeadConst make_head_const(int64_t v, int64_t off) {
    HeadConst c;
    const uint64_t va = v < 0 ? 0ull - (uint64_t)v : (uint64_t)v;
    // One call of the compiler's own 64-bit division per divisor.
    const uint64_t m = va ? (~0ull) / va : 0ull;
    uint64_t d = 0;
    if (va) {
        // 2^63 mod |v| by the same Barrett step: for a = 2^63 the estimate
        // floor(a * m / 2^64) is m >> 1.
        uint64_t r = (1ull << 63) - (m >> 1) * va;
        if (r >= va) r -= va;
        d = va - r;
    }
    uint32_t kind = 0;
    if (v < 0) kind |= kHeadNegative;
    if (va == 0) kind |= kHeadZero;
    if (v > 0 && va <= (1ull << 29)) kind |= kHeadFast;
    c.fast = make_uint4((uint32_t)m, (uint32_t)(m >> 32), 0u - 2u * (uint32_t)va, (uint32_t)d);
    c.off = off;
    c.ext = make_uint4((uint32_t)(va >> 32), (uint32_t)(d >> 32), kind, (uint32_t)va);
    return c;
}

// A head's constants prepared once in global memory (ple_prepare_heads), so
// that a kernel loads them instead of dividing: three 16-byte words per head,
// {fast}, {ext}, {off low, off high, 0, 0} (PLE_HEAD_BYTES = 48).
__device__ __forceinline__ void store_head_const(void* heads, int64_t k, const HeadConst& c) {
    uint4* h = static_cast<uint4*>(heads) + 3 * k;
    h[0] = c.fast;
    h[1] = c.ext;
    h[2] = make_uint4((uint32_t)(uint64_t)c.off, (uint32_t)((uint64_t)c.off >> 32), 0u, 0u);
}

__device__ __forceinline__ HeadConst load_head_const(const void* heads, int64_t k) {
    const uint4* h = static_cast<const uint4*>(heads) + 3 * k;
    HeadConst c;
    c.fast = __ldg(h);
    c.ext = __ldg(h + 1);
    const uint4 o = __ldg(h + 2);
    c.off = (int64_t)(((uint64_t)o.y << 32) | o.x);
    return c;
}

// The signed mix in offset binary, split into 32-bit words.
struct OffsetBinary {
    uint32_t lo;
    uint32_t hi;
};

__device__ __forceinline__ OffsetBinary offset_binary(uint64_t mix) {
    OffsetBinary u;
    u.lo = (uint32_t)mix;
    u.hi = (uint32_t)(mix >> 32) ^ 0x80000000u;
    return u;
}

// floormod(x, v) for 0 < v <= 2^29 from x's offset binary u, given
// c = {m_lo, m_hi, -2v, D} and nv = -v (mod 2^32; the caller derives it
// once per head by an arithmetic shift of -2v).  With -2v, the constant the
// first two corrections add, in the loaded word rather than computed, those
// adds no longer go to the integer-multiply pipe (measured on GB300: 1.4
// fewer multiply-pipe instructions per row id, the ALU count unchanged, so
// they fuse into the min).  The quotient estimate
// keeps only the three partial products that reach bits 64..95 of u*m and
// drops the carry out of bits 32..63 (at most 2), so it can fall 3 short of
// floor(u/v): the remainder estimate lies in [0, 4v), plus D in [1, 5v) <
// 2^32, and three conditional subtractions (2v, 2v, v) finish it.  The
// partial products are summed inside the multiplies (mul.hi, mad.hi,
// mad.lo) and each correction is min(r + (-k), r) on unsigned values.
// The body; with kAlu the sign-fix add is issued on the ALU (see
// floormod_fast_alu), taken where the last multiply needs it.
template <bool kAlu>
__device__ __forceinline__ uint32_t floormod_fast_body(OffsetBinary u, uint4 c, uint32_t nv,
                                                       uint32_t ones) {
    uint32_t t1, t2, q, r;
    asm("mul.hi.u32 %0, %1, %2;" : "=r"(t1) : "r"(u.lo), "r"(c.y));
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(t2) : "r"(u.hi), "r"(c.x), "r"(t1));
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(q) : "r"(u.hi), "r"(c.y), "r"(t2));
    const uint32_t lo_d = kAlu ? min(u.lo + c.w, ones) : u.lo + c.w;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(nv), "r"(lo_d));
    r = min(r + c.z, r);  // in [1, 5v): subtract 2v if it stays non-negative
    r = min(r + c.z, r);
    r = min(r + nv, r);  // and v
    return r;
}

__device__ __forceinline__ uint32_t floormod_fast(OffsetBinary u, uint4 c, uint32_t nv) {
    return floormod_fast_body<false>(u, c, nv, 0u);
}

// The same remainder with the sign-fix add issued on the integer ALU.  The
// compiler issues a plain 32-bit add as IMAD.IADD on the integer-multiply
// pipe, which the remainder's four multiplies already load; `ones` is
// 0xFFFFFFFF from a kernel parameter, so min(u.lo + D, ones) is the same sum,
// but the compiler cannot fold the min away and issues one add-min
// (VIADDMNMX) on the ALU.  Measured on GB300 where the multiply pipe bounds
// the kernel (int32 row ids): 1.5-4 % faster a call.
__device__ __forceinline__ uint32_t floormod_fast_alu(OffsetBinary u, uint4 c, uint32_t nv,
                                                      uint32_t ones) {
    return floormod_fast_body<true>(u, c, nv, ones);
}

__device__ __forceinline__ int64_t row_fast(OffsetBinary u, uint4 c, int64_t off) {
    return (int64_t)((uint64_t)off + floormod_fast(u, c, (uint32_t)((int32_t)c.z >> 1)));
}

// floormod(x, v) + off for any head.
__device__ __forceinline__ int64_t row_general(OffsetBinary u, uint4 c, int64_t off, uint4 ext) {
    if (ext.z & kHeadZero) return off;
    const uint64_t a = ((uint64_t)u.hi << 32) | u.lo;
    const uint64_t m = ((uint64_t)c.y << 32) | c.x;
    const uint64_t va = ((uint64_t)ext.x << 32) | ext.w;
    const uint64_t d = ((uint64_t)ext.y << 32) | c.w;
    const uint64_t q = __umul64hi(a, m);
    uint64_t r = a - q * va;  // [0, 2|v|)
    if (r >= va) r -= va;     // u mod |v|
    r += d;                   // [1, 2|v|), no wrap: at most 2^64 - 1
    if (r >= va) r -= va;     // floormod(x, |v|)
    if (ext.z & kHeadNegative) r = r ? r - va : 0;
    return (int64_t)(r + (uint64_t)off);
}

}  // namespace ple
