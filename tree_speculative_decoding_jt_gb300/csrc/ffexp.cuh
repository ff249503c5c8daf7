// ffexp.cuh -- accurate exp(x) for x <= 0 returned as an unevaluated sum of
// two floats (hi + lo), from fp32 arithmetic only.
//
// Used by the log-sum-exp of the draft rows, which must agree with an fp64
// reference to ~1e-11 relative while running at fp32 ALU rates (GB300's
// fp64 rate is far too low for one fp64 exp per vocabulary entry).
//
// Method: P. T. P. Tang, "Table-driven implementation of the exponential
// function in IEEE floating-point arithmetic", ACM TOMS 15(2), 1989:
//   x = k*ln2/64 + r,  exp(x) = 2^(k>>6) * 2^((k&63)/64) * exp(r),
// with the reduction constant ln2/64 split into C1 + C2 + C3 (C1, C2 with
// 10 significant bits so that k*C1 and k*C2 are exact for |k| < 2^14), the
// 64 table values 2^(j/64) held as float pairs (computed on the host in
// long double), and exp(r) - 1 = r + r^2/2 + r^3/6 + r^4/24 + r^5/120 for
// |r| <= ln2/128 (truncation error below 4e-17).  The linear term and the
// table product stay exact through FMA-based error-free transforms.
// Inputs below -87 return 0 (the caller's terms are relative to a maximum of
// 1, so they are below 2^-125 of the sum).
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>
#ifdef __CUDACC__
#define JT_HD __host__ __device__ __forceinline__
#else
#define JT_HD inline
#endif

namespace jt {

struct ffloat {
    float hi, lo;
};

// ln2/64 = C1 + C2 + C3 (+ 1.4e-18)
constexpr float kExpC1 = 0.010833740234375f;          // 0x1.63p-7
constexpr float kExpC2 = -3.3155083656311035e-06f;    // -0x1.bdp-19
constexpr float kExpC3 = -2.976022206446771e-11f;     // -0x1.05c61p-35
constexpr float kExpInvL = 92.33248138427734f;        // 64/ln2 (fp32)

JT_HD float jt_fmaf(float a, float b, float c) {
#ifdef __CUDA_ARCH__
    return __fmaf_rn(a, b, c);
#else
    return std::fmaf(a, b, c);
#endif
}

// Rounded multiply / add that the compiler may not fuse into an FMA (the
// error-free transforms below depend on each product being rounded).
JT_HD float jt_mul(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}

JT_HD float jt_add(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}

JT_HD float jt_pow2i(int n) {  // 2^n for -126 <= n <= 127
    uint32_t u = static_cast<uint32_t>(n + 127) << 23;
#ifdef __CUDA_ARCH__
    return __uint_as_float(u);
#else
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
#endif
}

JT_HD uint32_t jt_float_bits(float f) {
#ifdef __CUDA_ARCH__
    return __float_as_uint(f);
#else
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return u;
#endif
}

// 1.5 * 2^23: adding it to |v| < 2^22 leaves round-to-nearest(v) in the low
// mantissa bits, so the reduction needs no float-to-int conversion.
constexpr float kRoundMagic = 12582912.0f;

// exp(xh + xl) for finite xh >= -87, with xl a small correction
// (|xl| <= ulp(xh)).  tab_hi/tab_lo: 2^(j/64), j = 0..63, as float pairs.
JT_HD ffloat ffexp_in_range(float xh, float xl, const float* tab_hi, const float* tab_lo) {
    ffloat res;
    // k = nearest integer to xh * 64/ln2 (|k| < 2^13)
    const float tk = jt_fmaf(xh, kExpInvL, kRoundMagic);
    const float kf = jt_add(tk, -kRoundMagic);
    const int k = static_cast<int>(jt_float_bits(tk)) - 0x4B400000;
    const float r1 = jt_fmaf(-kf, kExpC1, xh);   // exact
    const float rh = jt_fmaf(-kf, kExpC2, r1);   // exact
    const float rl = jt_fmaf(-kf, kExpC3, xl);   // |rl| < 4e-7
    const float rc = jt_add(rh, rl);
    // p = rc^2/2 + rc^3/6 + rc^4/24 + rc^5/120
    float p = jt_fmaf(rc, 1.0f / 120.0f, 1.0f / 24.0f);
    p = jt_fmaf(rc, p, 1.0f / 6.0f);
    p = jt_fmaf(rc, p, 0.5f);
    p = (rc * rc) * p;
    const float q = rl + p;  // exp(r) = 1 + rh + q
    const int j = k & 63;
    const int n = k >> 6;  // floor division
    const float th = tab_hi[j], tl = tab_lo[j];
    // T*(1 + rh + q) = th + th*rh + (th*q + tl*(1 + rh))
    const float prod = jt_mul(th, rh);
    const float perr = jt_fmaf(th, rh, -prod);
    const float small = jt_fmaf(th, q, jt_fmaf(tl, rh, tl) + perr);
    const float s = jt_add(th, prod);  // |th| > |prod|: Fast2Sum
    const float e = jt_add(jt_add(th, -s), prod);
    const float sc = jt_pow2i(n);
    res.hi = jt_mul(s, sc);
    res.lo = jt_mul(jt_add(e, small), sc);
    return res;
}

// exp(xh + xl) for any xh <= 0: 0 below -87 and for -inf or NaN.
JT_HD ffloat ffexp(float xh, float xl, const float* tab_hi, const float* tab_lo) {
    if (!(xh >= -87.0f)) {  // also catches NaN and -inf
        ffloat res;
        res.hi = 0.0f;
        res.lo = 0.0f;
        return res;
    }
    return ffexp_in_range(xh, xl, tab_hi, tab_lo);
}

// Fill the 64-entry table 2^(j/64) = hi + lo (host side).
inline void ffexp_table(float* hi, float* lo) {
    for (int j = 0; j < 64; ++j) {
        long double v = exp2l(static_cast<long double>(j) / 64.0L);
        float h = static_cast<float>(v);
        hi[j] = h;
        lo[j] = static_cast<float>(v - static_cast<long double>(h));
    }
}

// Error-free sum of two floats: a + b = s + e exactly.
JT_HD void two_sum(float a, float b, float& s, float& e) {
    s = jt_add(a, b);
    const float bb = jt_add(s, -a);
    e = jt_add(jt_add(a, -jt_add(s, -bb)), jt_add(b, -bb));
}

// Float-float (unevaluated sum hi + lo) arithmetic from error-free
// transforms (Dekker / Knuth): |lo| <= ulp(hi)/2 after normalisation.
JT_HD ffloat ff_norm(float a, float b) {  // requires |a| >= |b| or a == 0
    ffloat r;
    r.hi = jt_add(a, b);
    r.lo = jt_add(b, -jt_add(r.hi, -a));
    return r;
}

JT_HD ffloat ff_add(ffloat a, ffloat b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e = jt_add(e, jt_add(a.lo, b.lo));
    return ff_norm(s, e);
}

JT_HD ffloat ff_mul(ffloat a, ffloat b) {
    const float p = jt_mul(a.hi, b.hi);
    float e = jt_fmaf(a.hi, b.hi, -p);
    e = jt_fmaf(a.hi, b.lo, jt_fmaf(a.lo, b.hi, e));
    return ff_norm(p, e);
}

}  // namespace jt
