// CPU checks of the kernels' RoPE angle reduction (rope_math.cuh) against the
// angle pos * theta^(-2k/r) of the Spark-X2.5 architecture page, §4, evaluated
// in long double.  Built and driven by test_rope_math.py.
#include <cmath>
#include <cstdint>

#include "rope_math.cuh"

namespace {
const long double kTwoPiL = 6.283185307179586476925286766559005768L;
}  // namespace

extern "C" {

// Largest error, in radians, of rope_turns over pairs k < r/2 and positions
// 0..pos_max in steps of `stride` (plus pos_max itself), with the frequency
// table built as the library builds it: u_k = theta^(-2k/r) / (2 pi) in fp64,
// split into fp32 hi + lo.  The reduced angle must also stay within 3/4
// turns of zero; a value outside counts as an error of 1 rad.
double rope_max_err(double theta, int r, int pos_max, int stride) {
    double worst = 0.0;
    for (int k = 0; k < r / 2; ++k) {
        const double inv = std::pow(theta, -2.0 * k / r);
        const double u = inv / 6.283185307179586476925286766559;
        const float hi = static_cast<float>(u);
        const float lo = static_cast<float>(u - static_cast<double>(hi));
        for (long long p = 0;; p = (p + stride < pos_max) ? p + stride : pos_max) {
            const float t = spark::rope_turns(static_cast<int>(p), hi, lo);
            const long double exact =
                static_cast<long double>(p) *
                std::pow(static_cast<long double>(theta), -2.0L * k / r) / kTwoPiL;
            long double d = static_cast<long double>(t) - exact;
            d -= std::nearbyint(d);  // the angle is defined modulo one turn
            double e = static_cast<double>(std::fabs(d) * kTwoPiL);
            if (!(std::fabs(t) <= 0.75f)) e = 1.0;
            if (!(e <= worst)) worst = e;  // NaN propagates
            if (p == pos_max) break;
        }
    }
    return worst;
}

}  // extern "C"
