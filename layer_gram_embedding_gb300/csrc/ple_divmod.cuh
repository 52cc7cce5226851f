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
//   m <= (2^64-1)/d gives a*m/2^64 < a/d.  So r' = a - q'*d lies in [0, 2d)
//   and one conditional subtraction yields a mod d.
//
//   When d <= 2^31, r' < 2^32, so r' equals the low 32 bits of a - q'*d and
//   only the low 32 bits of q' are needed: bits 64..95 of the 128-bit
//   product a*m, which take four 32-bit partial products and one carry.
//
// The sign rule on top: with r = |x| mod |v|,
//   v > 0: floormod(x, v) = r            if x >= 0,  (r ? |v| - r : 0) if x < 0
//   v < 0: floormod(x, v) = -floormod(-x, |v|), i.e. the same with the
//          condition flipped and the result negated.
#pragma once

#include <stdint.h>

namespace ple {

enum : uint32_t {
    kHeadNegative = 1u,  // vocab < 0
    kHeadZero = 2u,      // vocab == 0: the row is the offset
    kHeadFast = 4u,      // 0 < |vocab| <= 2^31: 32-bit remainder path
};

// One head's divisor constants, 32 bytes, laid out so the fast path's fields
// come in one 16-byte shared-memory load.
struct __align__(16) HeadConst {
    uint32_t m_lo;   // low / high words of m = floor((2^64 - 1) / |v|)
    uint32_t m_hi;
    uint32_t v_lo;   // |v| when it fits 32 bits
    uint32_t kind;   // kHead* flags
    int64_t off;     // the head's row offset
    uint64_t v_abs;  // |v| (2^63 for INT64_MIN)
};

__host__ __device__ __forceinline__ HeadConst make_head_const(int64_t v, int64_t off) {
    HeadConst c;
    const uint64_t va = v < 0 ? 0ull - (uint64_t)v : (uint64_t)v;
    // One call of the compiler's own 64-bit division per divisor.
    const uint64_t m = va ? (~0ull) / va : 0ull;
    uint32_t kind = 0;
    if (v < 0) kind |= kHeadNegative;
    if (va == 0) kind |= kHeadZero;
    if (va != 0 && va <= (1ull << 31)) kind |= kHeadFast;
    c.m_lo = (uint32_t)m;
    c.m_hi = (uint32_t)(m >> 32);
    c.v_lo = (uint32_t)va;
    c.kind = kind;
    c.off = off;
    c.v_abs = va;
    return c;
}

// a mod d for d <= 2^31, a < 2^64 (Barrett, low word only).
__device__ __forceinline__ uint32_t mod_small(uint64_t a, uint32_t d, uint32_t m0, uint32_t m1) {
    const uint32_t a0 = (uint32_t)a;
    const uint32_t a1 = (uint32_t)(a >> 32);
    const uint64_t p01 = (uint64_t)a0 * m1;
    const uint64_t p10 = (uint64_t)a1 * m0;
    const uint64_t mid = (uint64_t)__umulhi(a0, m0) + (uint32_t)p01 + (uint32_t)p10;
    const uint32_t q_lo = a1 * m1 + (uint32_t)(p01 >> 32) + (uint32_t)(p10 >> 32) +
                          (uint32_t)(mid >> 32);
    const uint32_t r = a0 - q_lo * d;
    return r >= d ? r - d : r;
}

// a mod d for any d >= 1, a < 2^64 (Barrett, full width).
__device__ __forceinline__ uint64_t mod_wide(uint64_t a, uint64_t d, uint64_t m) {
    const uint64_t q = __umul64hi(a, m);
    const uint64_t r = a - q * d;
    return r >= d ? r - d : r;
}

// |x| as an unsigned value and its sign; shared by every head of one order.
struct Magnitude {
    uint64_t a;
    bool neg;
};

__device__ __forceinline__ Magnitude magnitude(int64_t x) {
    Magnitude r;
    r.neg = x < 0;
    r.a = r.neg ? 0ull - (uint64_t)x : (uint64_t)x;
    return r;
}

// floormod(x, v) + off for the common case 0 < v <= 2^31.
__device__ __forceinline__ int64_t row_fast_positive(const Magnitude& x, uint32_t m0, uint32_t m1,
                                                     uint32_t v, int64_t off) {
    const uint32_t r = mod_small(x.a, v, m0, m1);
    const uint32_t t = (x.neg && r != 0u) ? v - r : r;
    return (int64_t)((uint64_t)off + (uint64_t)t);
}

// floormod(x, v) + off for any head.
__device__ __forceinline__ int64_t row_general(const Magnitude& x, const HeadConst& c) {
    uint64_t r;
    if (c.kind & kHeadZero) {
        r = 0;
    } else if (c.kind & kHeadFast) {
        r = mod_small(x.a, c.v_lo, c.m_lo, c.m_hi);
    } else {
        r = mod_wide(x.a, c.v_abs, ((uint64_t)c.m_hi << 32) | c.m_lo);
    }
    const bool vneg = (c.kind & kHeadNegative) != 0;
    const uint64_t t = ((x.neg != vneg) && r != 0) ? c.v_abs - r : r;
    const uint64_t res = vneg ? 0ull - t : t;
    return (int64_t)(res + (uint64_t)c.off);
}

}  // namespace ple
