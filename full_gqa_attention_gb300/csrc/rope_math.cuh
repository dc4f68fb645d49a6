// rope_math.cuh -- the RoPE angle arithmetic of the kernels: cos and sin of
// pos * theta^(-2k/r) for an integer position.  The kernels and the CPU tests
// compile this same header, so the tests check exactly the arithmetic the
// kernels run.
//
// Spark-X2.5 architecture (4B / 1.7B), §4 layered RoPE: full layers rotate the
// first 64 dims with theta = 5e6, sliding layers all 256 dims with theta = 1e4;
// pair k of a head turns by pos * theta^(-2k/r).
//
// The angle is carried in turns (1 turn = 2 pi rad) and reduced exactly to
// [-1/2, 1/2]; sin and cos of the reduced angle come from a quadrant split and
// the Taylor series of sin and cos at 0, on |x| <= pi/4 where the first
// omitted terms are below 2e-9.
#pragma once

#if defined(__CUDACC__)
#define SPARK_RM __host__ __device__ __forceinline__
#else
#include <cmath>
#define SPARK_RM inline
#endif

namespace spark {

// Correctly rounded fp32 operations, never fused with their neighbours (the
// exact reduction below relies on each rounding happening where written).
SPARK_RM float rm_mul(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    volatile float r = a * b;
    return r;
#endif
}

SPARK_RM float rm_add(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    volatile float r = a + b;
    return r;
#endif
}

SPARK_RM float rm_fma(float a, float b, float c) {
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return std::fma(a, b, c);
#endif
}

SPARK_RM float rm_rint(float x) {
#if defined(__CUDA_ARCH__)
    return rintf(x);
#else
    return std::nearbyint(x);
#endif
}

// (2 pi)^k / k!, the Taylor coefficients of sin(2 pi r) and cos(2 pi r) in r.
namespace rm {
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double p2 = kTwoPi * kTwoPi, p3 = p2 * kTwoPi, p4 = p3 * kTwoPi, p5 = p4 * kTwoPi;
constexpr double p6 = p5 * kTwoPi, p7 = p6 * kTwoPi, p8 = p7 * kTwoPi, p9 = p8 * kTwoPi;
constexpr double p10 = p9 * kTwoPi;
constexpr float S1 = static_cast<float>(kTwoPi);
constexpr float S3 = static_cast<float>(-p3 / 6.0);
constexpr float S5 = static_cast<float>(p5 / 120.0);
constexpr float S7 = static_cast<float>(-p7 / 5040.0);
constexpr float S9 = static_cast<float>(p9 / 362880.0);
constexpr float C2 = static_cast<float>(-p2 / 2.0);
constexpr float C4 = static_cast<float>(p4 / 24.0);
constexpr float C6 = static_cast<float>(-p6 / 720.0);
constexpr float C8 = static_cast<float>(p8 / 40320.0);
constexpr float C10 = static_cast<float>(-p10 / 3628800.0);
}  // namespace rm

// s = sin(2 pi t), c = cos(2 pi t) for |t| <= 1/2 (a little beyond is fine).
// t = q/4 + r with q = rint(4t) and |r| <= 1/8 (r exact: q/4 and t are both
// multiples of t's ulp); then 2 pi t = q pi/2 + x with |x| <= pi/4.
SPARK_RM void sincos_turns(float t, float &s, float &c) {
    const float q = rm_rint(rm_mul(4.0f, t));
    const float r = rm_fma(q, -0.25f, t);
    const float r2 = rm_mul(r, r);
    float sp = rm::S9;
    sp = rm_fma(sp, r2, rm::S7);
    sp = rm_fma(sp, r2, rm::S5);
    sp = rm_fma(sp, r2, rm::S3);
    sp = rm_fma(sp, r2, rm::S1);
    const float sx = rm_mul(sp, r);  // sin x
    float cp = rm::C10;
    cp = rm_fma(cp, r2, rm::C8);
    cp = rm_fma(cp, r2, rm::C6);
    cp = rm_fma(cp, r2, rm::C4);
    cp = rm_fma(cp, r2, rm::C2);
    const float cx = rm_fma(cp, r2, 1.0f);  // cos x
    // quadrant: sin(x + q pi/2), cos(x + q pi/2)
    const int iq = static_cast<int>(q) & 3;
    const float a = (iq & 1) ? cx : sx;
    const float b = (iq & 1) ? sx : cx;
    s = (iq & 2) ? -a : a;
    c = ((iq + 1) & 2) ? -b : b;
}

// The RoPE angle of one pair at an integer position, in turns, reduced to
// [-1/2, 1/2].
//
// The angle pos * inv_freq reaches 1e6 rad at the 1M-token positions of the
// full layers, where a plain fp32 product is off by up to ~0.03 rad.  Instead
// the angle is taken in turns and reduced exactly: with fp = pos (exact below
// 2^24) and u = u_hi + u_lo the frequency in turns (an unevaluated fp32 sum,
// from fp64 on the host),
//   p = fl(fp * u_hi),  e = fp * u_hi - p  (exact, by fma),
//   p - rint(p)         (exact: p and its nearest integer share the exponent),
//   t = (p - rint(p)) + (fp * u_lo + e)   in [-1/2, 1/2] up to rounding,
// so only the last two roundings (~2^-25 turns, ~2e-7 rad) remain.
SPARK_RM float rope_turns(int pos, float u_hi, float u_lo) {
    const float fp = static_cast<float>(pos);
    const float p = rm_mul(fp, u_hi);
    const float e = rm_fma(fp, u_hi, -p);
    const float f = rm_add(p, -rm_rint(p));
    return rm_add(f, rm_fma(fp, u_lo, e));
}

// cos and sin of the RoPE angle with sincos_turns.
SPARK_RM void rope_cos_sin_turns(int pos, float u_hi, float u_lo, float &c, float &s) {
    sincos_turns(rope_turns(pos, u_hi, u_lo), s, c);
}

}  // namespace spark
