// Host build of the device header's Newton-Raphson reciprocal
// (pow2_recip in int_device.cuh), checked against the definition
// floor(c 2^(e+s) / v) by 64-bit host division: a strided sweep over every
// leading-32-bit divisor class, random divisors of every bit length 1..40,
// and both edges of each bit length, for the two (c, s) pairs the kernels use.
#include <stdio.h>
#include <stdlib.h>
#include "../deterministic_integer_only_gb300/csrc/int_device.cuh"

using detint::u64;

static u64 splitmix(u64* x) {
    u64 z = (*x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int main(int argc, char** argv) {
    const u64 stride = argc > 1 ? strtoull(argv[1], 0, 10) : 127;
    const int per_len = argc > 2 ? atoi(argv[2]) : 20000;
    const u64 pairs[2][2] = {{127, 16}, {1, 23}};
    long long cases = 0, bad = 0;
    u64 st = 20250101;
    for (int k = 0; k < 2; ++k) {
        const u64 c = pairs[k][0];
        const int s = (int)pairs[k][1];
        for (u64 d = 1ull << 31; d < (1ull << 32); d += stride) {
            ++cases;
            if (detint::pow2_recip(d, 32, c, s) != (c << (32 + s)) / d) ++bad;
        }
        const int emax = c == 1 ? 39 : 40;
        for (int e = 1; e <= emax; ++e) {
            for (int i = 0; i < per_len; ++i) {
                u64 v;
                if (i < 32) v = (1ull << (e - 1)) + (u64)i;
                else if (i < 64) v = (1ull << e) - 1 - (u64)(i - 32);
                else v = (1ull << (e - 1)) | (e > 1 ? splitmix(&st) & ((1ull << (e - 1)) - 1) : 0);
                if ((v >> e) != 0 || (v >> (e - 1)) == 0) continue;
                ++cases;
                const u64 q = detint::pow2_recip(v, e, c, s);
                const u64 ref = (c << (e + s)) / v;
                if (q != ref) {
                    if (bad < 8) printf("mismatch c=%llu s=%d v=%llu: %llu != %llu\n", c, s, v, q, ref);
                    ++bad;
                }
            }
        }
    }
    printf("cases %lld mismatches %lld\n", cases, bad);
    return bad != 0;
}
