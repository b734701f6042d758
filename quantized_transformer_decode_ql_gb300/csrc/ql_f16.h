// IEEE binary16 conversions and the q4_0 block quantiser, usable from host and device code.
// Written from the IEEE 754 definitions: round to nearest, ties to even.
#pragma once

#include <stdint.h>
#include <math.h>

#ifdef __CUDACC__
#define QL_HD __host__ __device__ __forceinline__
#else
#define QL_HD inline
#endif

namespace ql {

QL_HD uint64_t f64_bits(double x) {
    union { double d; uint64_t u; } c;
    c.d = x;
    return c.u;
}

// Nearest binary16 to x (ties to the even significand); overflow gives +-inf.
QL_HD uint16_t f64_to_f16_rne(double x) {
    const uint64_t b = f64_bits(x);
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    const uint64_t a = b & 0x7FFFFFFFFFFFFFFFull;
    if (a >= 0x7FF0000000000000ull)                      // inf or NaN
        return (uint16_t)(sign | 0x7C00u | (a > 0x7FF0000000000000ull ? 0x0200u : 0u));
    const int e = (int)(a >> 52) - 1023;                 // unbiased exponent
    if (e < -26) return sign;                            // below half the smallest subnormal
    const uint64_t mant = (a & 0x000FFFFFFFFFFFFFull) | 0x0010000000000000ull;  // 53 bits
    // value = mant * 2^(e-52). A normal f16 keeps 11 significant bits; a subnormal keeps
    // the bits at or above 2^-24.
    int shift = (e >= -14) ? 42 : (28 - e);              // bits of mant dropped
    uint64_t q = mant >> shift;
    const uint64_t rem = mant & ((1ull << shift) - 1);
    const uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1;
    if (e >= -14) {
        int ee = e;
        if (q == (1ull << 11)) { q >>= 1; ee += 1; }      // rounding carried into the exponent
        if (ee > 15) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | (uint16_t)((ee + 15) << 10) | (uint16_t)(q & 0x3FFu));
    }
    // subnormal (q <= 0x400; q == 0x400 is exactly the smallest normal, same bit pattern)
    return (uint16_t)(sign | (uint16_t)q);
}

QL_HD double f16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int ex = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    double v;
    if (ex == 0) v = ldexp((double)m, -24);
    else if (ex == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m | 0x400), ex - 25);
    return sign ? -v : v;
}

// Round half to even, for |v| < 2^52.
QL_HD double round_half_even(double v) {
    double r = floor(v);
    const double f = v - r;
    if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return r;
}

// One q4_0 block: 32 f32 weights -> f16 scale bits and 16 code bytes.
// d = f16(max|x| / 7); q = clamp(rhe(x / d), -7, 7) + 8; byte j = q[j] | q[j+16] << 4.
// Returns 0, 1 for a non-finite weight, 2 for a scale that overflows f16 (both leave
// d = 0, q = 8).
QL_HD int q4_0_block(const float* x, uint16_t* scale, uint8_t* quants) {
    double amax = 0.0;
    int bad = 0;
    for (int e = 0; e < 32; ++e) {
        const double v = (double)x[e];
        if (!(fabs(v) <= 1.7976931348623157e308)) bad = 1;   // NaN or inf
        const double av = fabs(v);
        if (av > amax) amax = av;
    }
    uint16_t d16 = bad ? (uint16_t)0 : f64_to_f16_rne(amax / 7.0);
    if (!bad && (d16 & 0x7C00u) == 0x7C00u) { bad = 2; d16 = 0; }
    const double d = f16_to_f64(d16);
    uint8_t c[32];
    for (int e = 0; e < 32; ++e) {
        int q = 8;
        if (d > 0.0) {
            double r = round_half_even((double)x[e] / d);
            r = r < -7.0 ? -7.0 : (r > 7.0 ? 7.0 : r);
            q = (int)r + 8;
        }
        c[e] = (uint8_t)q;
    }
    for (int j = 0; j < 16; ++j) quants[j] = (uint8_t)(c[j] | (c[j + 16] << 4));
    *scale = d16;
    return bad;
}

}  // namespace ql
