// Host-side accuracy check of the library's table-driven exp (ffexp.cuh),
// compiled with g++ -ffp-contract=off so that every operation rounds as the
// device code does (the device code uses explicit FMA / non-fused intrinsics).
// Prints: max relative error, count of inexact reductions, samples.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <random>

#include "../../tree_speculative_decoding_jt_gb300/csrc/ffexp.cuh"

int main() {
    float th[64], tl[64];
    jt::ffexp_table(th, tl);
    std::mt19937_64 rng(12345);
    std::uniform_real_distribution<double> U(-87.0, 0.0);
    double max_rel = 0.0;
    long inexact = 0, n = 0;
    auto check = [&](float xh, float xl) {
        const float kf = std::nearbyintf(xh * jt::kExpInvL);
        // exactness of the two-step reduction
        const double exact_r = (double)xh - (double)kf * (double)jt::kExpC1 - (double)kf * (double)jt::kExpC2;
        const float r1 = std::fmaf(-kf, jt::kExpC1, xh);
        const float rh = std::fmaf(-kf, jt::kExpC2, r1);
        if ((double)rh != exact_r) ++inexact;
        jt::ffloat y = jt::ffexp(xh, xl, th, tl);
        long double ref = expl((long double)xh + (long double)xl);
        long double got = (long double)y.hi + (long double)y.lo;
        // relative error while the low part stays a normal float; below
        // x = -72 only the absolute error matters (the caller's terms are
        // relative to a maximum term of 1) and it must stay below 1e-30
        double rel = (double)fabsl((got - ref) / ref);
        if (xh < -72.0f) rel = (double)fabsl(got - ref) > 1e-30 ? 1.0 : 0.0;
        if (rel > max_rel) max_rel = rel;
        ++n;
    };
    for (int i = 0; i < 4000000; ++i) {
        float xh = (float)U(rng);
        float xl = (float)((U(rng) / 87.0) * 1e-7 * std::fabs(xh));
        if (xh + xl > 0 || xh + xl < -87) xl = 0;
        check(xh, xl);
    }
    // dense sweep near 0 and around every table boundary
    for (float x = -1e-3f; x <= 0.0f; x += 3.7e-9f) check(x, 0.0f);
    for (int k = -8000; k <= 0; ++k) {
        float c = (float)(k * (0.6931471805599453 / 64.0));
        for (int d = -4; d <= 4; ++d) check(std::nextafterf(c, d < 0 ? -100.f : 100.f) + d * 1e-7f * (1 + std::fabs(c)), 0.0f);
    }
    // two_sum is error-free
    long ts_bad = 0;
    std::uniform_real_distribution<double> V(-1e3, 1e3);
    for (int i = 0; i < 1000000; ++i) {
        float a = (float)V(rng), b = (float)(V(rng) * 1e-4);
        float s, e;
        jt::two_sum(a, b, s, e);
        if ((long double)s + e != (long double)a + b) ++ts_bad;
    }
    printf("max_rel %.3e inexact_reductions %ld samples %ld two_sum_bad %ld\n", max_rel, inexact, n, ts_bad);
    return (max_rel < 1e-11 && inexact == 0 && ts_bad == 0) ? 0 : 1;
}
