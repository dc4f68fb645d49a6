// CPU checks of the kernels' RoPE angle arithmetic (rope_math.cuh) against
// the angle pos * theta^(-2k/r) of the Spark-X2.5 architecture page, §4,
// evaluated in long double.  Built and driven by test_rope_math.py.
#include <cmath>
#include <cstdint>

#include "rope_math.cuh"

namespace {

const long double kTwoPiL = 6.283185307179586476925286766559005768L;

// sin and cos of 2 pi t with t in turns, in long double.
void exact_turns(long double t, long double &s, long double &c) {
    t -= std::nearbyint(t);
    s = std::sin(kTwoPiL * t);
    c = std::cos(kTwoPiL * t);
}

// splitmix64: a fixed sequence of test points
uint64_t next(uint64_t &x) {
    uint64_t z = (x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace

extern "C" {

// Largest |error| of sincos_turns over n evenly spaced points of [-1/2, 1/2],
// the quadrant edges and n random points.
double sincos_turns_max_err(int n) {
    double worst = 0.0;
    auto check = [&](float t) {
        float s, c;
        spark::sincos_turns(t, s, c);
        long double es, ec;
        exact_turns(t, es, ec);
        const double e = std::fmax(std::fabs(static_cast<double>(s - es)),
                                   std::fabs(static_cast<double>(c - ec)));
        if (!(e <= worst)) worst = e;  // NaN propagates
    };
    for (int i = 0; i <= n; ++i) check(-0.5f + static_cast<float>(i) / n);
    for (int q = -4; q <= 4; ++q) {
        const float edge = q / 8.0f;
        check(edge);
        check(std::nextafter(edge, 1.0f));
        check(std::nextafter(edge, -1.0f));
    }
    uint64_t x = 12345;
    for (int i = 0; i < n; ++i)
        check(static_cast<float>(static_cast<double>(next(x) >> 11) * 0x1.0p-53 - 0.5));
    return worst;
}

// Largest |error| of rope_cos_sin_turns over pairs k < r/2 and positions
// 0..pos_max in steps of `stride` (plus pos_max itself), with the frequency
// table built as the library builds it: u_k = theta^(-2k/r) / (2 pi) in fp64,
// split into fp32 hi + lo.
double rope_max_err(double theta, int r, int pos_max, int stride) {
    double worst = 0.0;
    for (int k = 0; k < r / 2; ++k) {
        const double inv = std::pow(theta, -2.0 * k / r);
        const double u = inv / 6.283185307179586476925286766559;
        const float hi = static_cast<float>(u);
        const float lo = static_cast<float>(u - static_cast<double>(hi));
        for (long long p = 0; p <= pos_max; p += (p + stride > pos_max && p != pos_max)
                                                     ? (pos_max - p) : stride) {
            float c, s;
            spark::rope_cos_sin_turns(static_cast<int>(p), hi, lo, c, s);
            const long double turns =
                static_cast<long double>(p) * std::pow(static_cast<long double>(theta),
                                                       -2.0L * k / r) / kTwoPiL;
            long double es, ec;
            exact_turns(turns, es, ec);
            const double e = std::fmax(std::fabs(static_cast<double>(s - es)),
                                       std::fabs(static_cast<double>(c - ec)));
            if (!(e <= worst)) worst = e;
            if (p == pos_max) break;
        }
    }
    return worst;
}

}  // extern "C"
