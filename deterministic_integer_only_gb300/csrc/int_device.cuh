// Integer primitives for the detint kernels. The scalar routines also build
// for the host (tests compare that build with the oracle); the warp-
// cooperative forms at the end are device-only.
//
// Every rule here is the frozen arithmetic of the integer-only forward pass:
// round-to-nearest shifts with ties toward +infinity, floor divisions of
// non-negative integers, floor square roots and 15-bit dyadic scales
// (DetLLM blog, section "DetLLM": every tensor carries a scale m/2^k, and
// rescaling is one integer multiply and one shift with a fixed rounding rule;
// DetLLM README, "Layout": intmath freezes the rounding rules).
//
// No floating-point type, literal or intrinsic appears in this file or in any
// kernel file, and there is no division or remainder by a value known only at
// run time: CUDA may lower those through a floating-point reciprocal, so
// divisions go through udiv64 below (restoring long division), its
// warp-parallel form, or pow2_recip (Newton-Raphson) for power-of-two
// numerators.
#pragma once
#include <stdint.h>

namespace detint {

typedef long long i64;
typedef unsigned long long u64;

// number of binary digits (bitlen(0) = 0)
__host__ __device__ __forceinline__ int bitlen_u64(u64 x) {
#ifdef __CUDA_ARCH__
    return 64 - __clzll((long long)x);
#else
    return x ? 64 - __builtin_clzll(x) : 0;    // host build of this header (tests)
#endif
}

// x / 2^s rounded to nearest, ties toward +infinity; s in [0, 62]
__host__ __device__ __forceinline__ i64 rshr(i64 x, int s) {
    return s <= 0 ? x : ((x + (1LL << (s - 1))) >> s);
}
__host__ __device__ __forceinline__ int rshr32(int x, int s) {
    return s <= 0 ? x : ((x + (1 << (s - 1))) >> s);
}
__host__ __device__ __forceinline__ i64 sat_b(i64 x, i64 b) { return x > b ? b : (x < -b ? -b : x); }
__host__ __device__ __forceinline__ int sat32(i64 x) { return (int)sat_b(x, 2147483647LL); }
__host__ __device__ __forceinline__ int sat127(i64 x) { return (int)sat_b(x, 127); }

// floor(n / d) for d >= 1, by restoring long division over the quotient bits
static __host__ __device__ __noinline__ u64 udiv64(u64 n, u64 d) {
    if (n < d) return 0;
    int sh = bitlen_u64(n) - bitlen_u64(d);
    u64 dd = d << sh;
    u64 q = 0;
    for (int i = sh; i >= 0; --i) {
        q <<= 1;
        if (n >= dd) { n -= dd; q |= 1ull; }
        dd >>= 1;
    }
    return q;
}

// floor(sqrt(n)), digit by digit
static __host__ __device__ __noinline__ u64 isqrt_u64(u64 n) {
    u64 r = 0, bit = 1ull << 62;
    while (bit > n) bit >>= 2;
    while (bit) {
        if (n >= r + bit) { n -= r + bit; r = (r >> 1) + bit; }
        else r >>= 1;
        bit >>= 2;
    }
    return r;
}

// floor(sqrt(n)) for n < 2^62 in one thread, by the Newton-Raphson
// reciprocal square root in integers: n is scaled by an even power of two
// to m in [2^60, 2^62); with f = m / 2^62 in [1/4, 1), y ~ 2^30 / sqrt(f)
// starts from the minimax line 2.132 - 1.218 f (relative error <= 0.087) and
// takes four steps y <- y (3 - f y^2) / 2 (all products below 2^64); then
// r = f y 2^31 is within a few units of sqrt(m), the exact checks r^2 <= m <
// (r + 1)^2 settle it, and sqrt(n) = floor(r / 2^(shift / 2))
__host__ __device__ __forceinline__ u64 isqrt_fast(u64 n) {
    if (n == 0) return 0;
    int s = 62 - bitlen_u64(n);
    s -= s & 1;
    const u64 m = n << s;                                    // [2^60, 2^62)
    const u64 m32 = m >> 30;                                 // [2^30, 2^32)
    u64 y = 2289217569ull - ((1307817542ull * m32) >> 32);   // Q30
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const u64 t = (m32 * ((y * y) >> 30)) >> 32;         // f y^2, Q30
        y = (y * (3221225472ull - t)) >> 31;
    }
    u64 r = (m32 * y) >> 31;
    for (int i = 0; i < 4 && r * r > m; ++i) --r;
    for (int i = 0; i < 4 && (r + 1) * (r + 1) <= m; ++i) ++r;
    return r >> (s >> 1);
}

// (m, k): m = round(N 2^k / D) (ties up) with 2^14 <= N 2^k / D < 2^15
static __host__ __device__ __noinline__ void dyadic_dev(u64 N, u64 D, int* m_out, int* k_out) {
    int k = 14 + bitlen_u64(D) - bitlen_u64(N);
    for (int it = 0; it < 4; ++it) {   // the estimate is within one of k
        u64 lhs, lo;
        if (k >= 0) { lhs = N << k; lo = D << 14; }
        else { lhs = N; lo = D << (14 - k); }
        if (lhs < lo) { ++k; continue; }
        if (lhs >= (lo << 1)) { --k; continue; }
        break;
    }
    u64 num, den;
    if (k >= 0) { num = (N << (k + 1)) + D; den = D << 1; }
    else { num = (N << 1) + (D << (-k)); den = D << (1 - k); }
    *m_out = (int)udiv64(num, den);
    *k_out = k;
}

// 2^(delta/1024) in Q15 for delta <= 0: a cubic on the fraction of the
// base-2 exponent (Horner form, one rounding shift per step) and a right
// shift for its integer part (DetLLM README, "Layout": DI-Exp)
__host__ __device__ __forceinline__ int exp2q_dev(i64 delta) {
    i64 ip = delta >> 10;                 // floor
    if (ip <= -24) return 0;
    int f = (int)(delta & 1023);
    int inner = 7419 + rshr32(2562 * f, 10);
    int mid = 22787 + rshr32(f * inner, 10);
    int p2 = 32768 + rshr32(f * mid, 10);
    return rshr32(p2, (int)(-ip));
}

// floor(c 2^(e+s) / v) for v >= 1 with e = bitlen(v) <= 40, c 2^(e+s) < 2^63
// and c 2^s < 2^30, s <= 30 (the quotient lies in (c 2^s, c 2^(s+1)]): the
// per-row quantisation multiplier (c = 127, s = 16) and the row-sum
// reciprocals (c = 1, s = 23). Newton-Raphson division (as in Goldschmidt's
// and Newton's reciprocal iterations, all in integers): d = the leading 32
// bits of v; y ~ 2^62 / d from the linear minimax seed 48/17 - 32/17 d' of
// 1/d' on [1/2, 1) (relative error <= 1/17) and three Newton steps
// y += y (2^62 - d y) / 2^62 in Q30 (error ~1/17 -> 2^-8 -> 2^-16 -> a few
// units of 2^-30), every product 32 x 32 bits; q = c y / 2^(30 - s) is then
// within one of the quotient (within one more when v has more than 32
// bits), and the exact remainder N - q v (one 64-bit product, |.| < 3 v)
// settles it by at most two steps each way.
__host__ __device__ __forceinline__ u64 pow2_recip(u64 v, int e, u64 c, int s) {
    const uint32_t d = (uint32_t)(e <= 32 ? v << (32 - e) : v >> (e - 32));   // [2^31, 2^32)
    uint32_t y = 3031741621u - (uint32_t)(((u64)2021161080u * d) >> 32);     // Q30, (0.94, 1.89] * 2^30
#pragma unroll
    for (int it = 0; it < 3; ++it) {
        const u64 p = (u64)d * y;                                             // ~2^62, < 2^63
        const bool over = p > (1ull << 62);
        const u64 t = over ? p - (1ull << 62) : (1ull << 62) - p;
        const uint32_t corr = (uint32_t)(((u64)y * (uint32_t)(t >> 31)) >> 31);
        y = over ? y - corr : y + corr;
    }
    const u64 N = c << (e + s);
    u64 q = (c * y) >> (30 - s);
    long long rem = (long long)(N - q * v);                                   // in (-2v, 3v)
    const long long vv = (long long)v;
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if (rem < 0) { --q; rem += vv; }
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (rem >= vv) { ++q; rem -= vv; }
    return q;
}

// floor(n / d) for d >= 1 when the quotient is below 2^31 and n < 2^63, by
// the Newton-Raphson reciprocal of d's leading 32 bits (the steps of
// pow2_recip), a 128-bit product n y and the exact remainder n - q d, which
// settles the estimate (within a few units) by single steps
__host__ __device__ __forceinline__ u64 udiv_small(u64 n, u64 d) {
    const int e = bitlen_u64(d);
    const uint32_t d32 = (uint32_t)(e <= 32 ? d << (32 - e) : d >> (e - 32));   // [2^31, 2^32)
    uint32_t y = 3031741621u - (uint32_t)(((u64)2021161080u * d32) >> 32);     // ~2^62 / d32, Q30
#pragma unroll
    for (int it = 0; it < 3; ++it) {
        const u64 p = (u64)d32 * y;
        const bool over = p > (1ull << 62);
        const u64 t = over ? p - (1ull << 62) : (1ull << 62) - p;
        const uint32_t corr = (uint32_t)(((u64)y * (uint32_t)(t >> 31)) >> 31);
        y = over ? y - corr : y + corr;
    }
    // n / d ~ n y / 2^(30 + e): the 128-bit product's bits from 30 + e up
    const int sh = 30 + e;                        // in [31, 94]
#ifdef __CUDA_ARCH__
    const u64 hi = __umul64hi(n, (u64)y);
#else
    const u64 hi = (u64)(((unsigned __int128)n * y) >> 64);
#endif
    const u64 lo = n * (u64)y;
    u64 q = sh >= 64 ? hi >> (sh - 64) : ((hi << (64 - sh)) | (lo >> sh));
    long long rem = (long long)(n - q * d);
    const long long dd = (long long)d;
    for (int i = 0; i < 4 && rem < 0; ++i) { --q; rem += dd; }
    for (int i = 0; i < 4 && rem >= dd; ++i) { ++q; rem -= dd; }
    return q;
}

// dyadic(N, D) in one thread: the exponent by bit lengths and comparisons,
// the mantissa by udiv_small (quotient <= 2^15)
__host__ __device__ __forceinline__ void dyadic_fast(u64 N, u64 D, int* m_out, int* k_out) {
    int k = 14 + bitlen_u64(D) - bitlen_u64(N);
    for (int it = 0; it < 4; ++it) {
        u64 lhs, lo;
        if (k >= 0) { lhs = N << k; lo = D << 14; }
        else { lhs = N; lo = D << (14 - k); }
        if (lhs < lo) { ++k; continue; }
        if (lhs >= (lo << 1)) { --k; continue; }
        break;
    }
    u64 num, den;
    if (k >= 0) { num = (N << (k + 1)) + D; den = D << 1; }
    else { num = (N << 1) + (D << (-k)); den = D << (1 - k); }
    *m_out = (int)udiv_small(num, den);
    *k_out = k;
}

// rshr(acc * M, s) with the product formed exactly in 128 bits, for the
// exact mode's int64 accumulators of 16-bit weights (|acc| < 2^36, M < 2^31,
// 1 <= s <= 100; the result must fit int64): the product as a two's-
// complement (hi, lo) pair from 32-bit partial products, plus 2^(s-1), then
// an arithmetic shift of the pair. The same code runs on host and device.
__host__ __device__ __forceinline__ i64 rshr_mul128(i64 acc, u64 M, int s) {
    const bool neg = acc < 0;
    const u64 a = neg ? (u64)(-acc) : (u64)acc;              // < 2^36
    const u64 a0 = a & 0xffffffffull, a1 = a >> 32, m0 = M & 0xffffffffull, m1 = M >> 32;
    const u64 p00 = a0 * m0, p01 = a0 * m1, p10 = a1 * m0, p11 = a1 * m1;
    const u64 mid = (p00 >> 32) + (p01 & 0xffffffffull) + (p10 & 0xffffffffull);
    u64 lo = (p00 & 0xffffffffull) | (mid << 32);
    u64 hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
    if (neg) {                                                // two's complement of (hi, lo)
        lo = ~lo + 1;
        hi = ~hi + (lo == 0 ? 1 : 0);
    }
    // + 2^(s-1)
    if (s - 1 < 64) {
        const u64 h = 1ull << (s - 1);
        const u64 nlo = lo + h;
        hi += nlo < lo ? 1 : 0;
        lo = nlo;
    } else {
        hi += 1ull << (s - 1 - 64);
    }
    // arithmetic shift right by s of the signed pair
    if (s < 64) return (i64)((lo >> s) | (hi << (64 - s)));
    return (i64)hi >> (s - 64);
}

// Q15 sigmoid of the SwiGLU gate from z = Q10 of |g| log2 e: with
// D = 2^15 + exp2q(-z), round(2^30 / D) = floor((2^31 + D) / 2D) <= 2^15,
// = 2^15 only for D = 2^15 (every z > 23552); otherwise 15 quotient bits by
// restoring division in 32 bits
__host__ __device__ __forceinline__ unsigned sigmoid_q15(i64 z) {
    const int Ez = exp2q_dev(-z);
    const unsigned D = 32768u + (unsigned)Ez;            // [2^15, 2^16]
    unsigned q = 32768u;
    if (D != 32768u) {
        unsigned num = 0x80000000u + D, dd = D << 15;   // 2D * 2^14 < 2^32
        q = 0;
#pragma unroll
        for (int i = 14; i >= 0; --i) {
            q <<= 1;
            if (num >= dd) { num -= dd; q |= 1u; }
            dd >>= 1;
        }
    }
    return q;
}

__host__ __device__ __forceinline__ i64 swiglu_z(int g) {
    const i64 ag = g < 0 ? -(i64)g : (i64)g;
    return rshr(ag * 47274LL, 17);
}

__host__ __device__ __forceinline__ int swiglu_finish(int g, int u, unsigned q) {
    const i64 sg = g >= 0 ? (i64)q : 32768LL - (i64)q;
    const i64 silu = rshr((i64)g * sg, 15);
    return sat32(rshr(silu * (i64)u, 14));
}

// one SwiGLU channel from saturated Q12 gate/up values (Q10 result)
__host__ __device__ __forceinline__ int swiglu_dev(int g, int u) {
    return swiglu_finish(g, u, sigmoid_q15(swiglu_z(g)));
}

// ------------------------------------------------ warp reductions
// max and sum over the 32 lanes of a warp on the redux unit, 64-bit values
// as 32-bit slices: the maximum of the high words, then of the low words of
// the lanes holding it; the sum modulo 2^64 as three sums of slices of 22,
// 22 and 20 bits, each total below 2^27
#if !defined(__CUDA_ARCH__) || __CUDA_ARCH__ >= 800
__device__ __forceinline__ u64 redux_max_u64(u64 v) {
    const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(v >> 32));
    const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(v >> 32) == hi ? (unsigned)v : 0u);
    return ((u64)hi << 32) | lo;
}
__device__ __forceinline__ u64 redux_sum_u64(u64 v) {
    const unsigned s0 = __reduce_add_sync(0xffffffffu, (unsigned)(v & 0x3fffffu));
    const unsigned s1 = __reduce_add_sync(0xffffffffu, (unsigned)((v >> 22) & 0x3fffffu));
    const unsigned s2 = __reduce_add_sync(0xffffffffu, (unsigned)(v >> 44));
    return (u64)s0 + ((u64)s1 << 22) + ((u64)s2 << 44);
}
#endif

}  // namespace detint
