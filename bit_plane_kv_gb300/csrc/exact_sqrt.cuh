// exact_sqrt.cuh -- IEEE binary64 square root, round to nearest, of a positive
// normal double, computed with 64-bit integer arithmetic from one fp32
// reciprocal-square-root seed.
//
// The plan's geometric bisection (Fathom §3.3: theta by a 30-step log
// bisection, mid = sqrt(lo * hi)) is a chain of 30 dependent square roots.
// The fp64 square root has a long latency on this part; this routine returns
// exactly the same bits (the correctly rounded root) in less time:
//   1. seed y ~ m^-1/2 from the fp32 rsqrt of the top 24 bits of the
//      mantissa m (relative error about 2^-22);
//   2. two coupled Newton steps (g -> sqrt(m), h -> 1 / (2 sqrt(m)):
//      r = 1/2 - g h, g += g r, h += h r) in 64-bit fixed point, which
//      leave the root within a few units of its last place;
//   3. the exact integer remainder M - r^2 moves r to floor(sqrt(M)), and
//      M - r^2 > r decides the rounding (a square root has no ties).
// Step 3 makes the result exact for any seed within the convergence range
// of step 2, so a host build (whose seed is 1 / sqrtf) computes the same
// bits and can be checked against the C library on the CPU.
#pragma once

#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define FATHOM_HD __host__ __device__ __forceinline__
#else
#define FATHOM_HD inline
#endif
#ifndef __CUDA_ARCH__
#include <cmath>
#endif

namespace fathom {
namespace xsqrt {

FATHOM_HD uint64_t umulhi(uint64_t a, uint64_t b) {
#ifdef __CUDA_ARCH__
    return __umul64hi(a, b);
#else
    return (uint64_t)(((unsigned __int128)a * b) >> 64);
#endif
}
FATHOM_HD int64_t smulhi(int64_t a, int64_t b) {
#ifdef __CUDA_ARCH__
    return __mul64hi(a, b);
#else
    return (int64_t)(((__int128)a * b) >> 64);
#endif
}
FATHOM_HD float rsqrt_seed(float f) {
#ifdef __CUDA_ARCH__
    float y;
    asm("rsqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(f));
    return y;
#else
    return 1.0f / std::sqrt(f);
#endif
}
FATHOM_HD uint32_t f2u(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}
FATHOM_HD float u2f(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}

// x: bits of a positive normal double.  seed_scale multiplies the seed (1 on
// the device; host tests perturb it to cover the device seed's error).
FATHOM_HD uint64_t sqrt_rn(uint64_t x, float seed_scale = 1.0f) {
    long long e = (long long)(x >> 52) - 1075;                // x = m * 2^e
    uint64_t m = (x & ((1ull << 52) - 1)) | (1ull << 52);
    if (e & 1) { m <<= 1; e -= 1; }                           // e even, m in [2^52, 2^54)
    // sqrt(x) = sqrt(M) * 2^((e - 52) / 2) with M = m * 2^52 in [2^104, 2^106)
    const int k = (int)((m >> 53) & 1);
    const float f = u2f(((uint32_t)(127 + 52 + k) << 23) | (uint32_t)((m >> (29 + k)) & 0x7fffff));
    const uint32_t yb = f2u(rsqrt_seed(f) * seed_scale);     // ~ m^-1/2, in about (2^-27, 2^-26]
    const uint64_t Y = (uint64_t)((yb & 0x7fffff) | 0x800000) << ((int)(yb >> 23) - 62);   // y * 2^88
    int64_t G = (int64_t)umulhi(m << 10, Y);                  // g * 2^34, g = m y
    int64_t H = (int64_t)Y;                                   // h * 2^89, h = y / 2
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int64_t R = ((int64_t)1 << 58) - (int64_t)umulhi((uint64_t)G, (uint64_t)H);   // (1/2 - g h) 2^59
        G += smulhi(G, R << 5);
        H += smulhi(H, R << 5);
    }
    uint64_t r = (uint64_t)G >> 8;                            // ~ sqrt(M), within a few units
    long long d = (long long)((m << 52) - r * r);             // M - r^2: small, the low 64 bits carry it
    while (d < 0) { d += (long long)(2 * r - 1); --r; }
    while (d > (long long)(2 * r)) { ++r; d -= (long long)(2 * r - 1); }
    if ((uint64_t)d > r) ++r;                                 // sqrt(M) >= r + 1/2
    long long be = (e - 52) / 2 + 1075;
    if (r >> 53) { r >>= 1; ++be; }
    return ((uint64_t)be << 52) | (r & ((1ull << 52) - 1));
}

}  // namespace xsqrt
}  // namespace fathom
