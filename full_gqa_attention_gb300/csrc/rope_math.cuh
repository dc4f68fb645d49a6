// rope_math.cuh -- the RoPE angle arithmetic of the kernels: the angle
// pos * theta^(-2k/r) of an integer position, in turns, reduced exactly to
// [-1/2, 1/2] (the kernels then take sincospif of twice it).  The kernels and
// the CPU tests compile this same header, so the tests check exactly the
// reduction the kernels run.
//
// Spark-X2.5 architecture (4B / 1.7B), §4 layered RoPE: full layers rotate the
// first 64 dims with theta = 5e6, sliding layers all 256 dims with theta = 1e4;
// pair k of a head turns by pos * theta^(-2k/r).
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

// The RoPE angle of one pair at an integer position, in turns, reduced to
// about [-1/2, 1/2].
//
// The angle pos * inv_freq reaches 1e6 rad at the 1M-token positions of the
// full layers, where a plain fp32 product is off by up to ~0.03 rad.  Instead
// the angle is taken in turns and reduced exactly: with fp = pos (exact below
// 2^24) and u = u_hi + u_lo the frequency in turns (an unevaluated fp32 sum,
// from fp64 on the host),
//   p = fl(fp * u_hi),  e = fp * u_hi - p  (exact, by fma),
//   p - rint(p)         (exact: p and its nearest integer share the exponent),
//   t = (p - rint(p)) + (fp * u_lo + e),
// so only the last two roundings (~2^-25 turns, ~2e-7 rad) remain.  The
// correction fp * u_lo + e is at most ulp(p), so |t| <= 3/4 for positions
// below 2^24 (sin and cos are periodic: no further reduction is needed).
SPARK_RM float rope_turns(int pos, float u_hi, float u_lo) {
    const float fp = static_cast<float>(pos);
    const float p = rm_mul(fp, u_hi);
    const float e = rm_fma(fp, u_hi, -p);
    const float f = rm_add(p, -rm_rint(p));
    return rm_add(f, rm_fma(fp, u_lo, e));
}

}  // namespace spark
