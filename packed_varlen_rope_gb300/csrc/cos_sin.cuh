// cos and sin of a binary32 angle, correctly rounded to binary32, without the FP64 pipe
// for all but about 4 angles in 100,000.
//
// The rotation needs c = RN32(cos phi) and s = RN32(sin phi) for phi = RN32(pos * w_j):
// the binary64 cosine and sine rounded once to binary32.  GB300 runs binary64 at a small
// fraction of its binary32 rate, so evaluating them in binary64 for every (position,
// frequency) pair makes a rotation without a cos/sin table compute-bound.  Instead:
//
//  1. Argument reduction (Cody and Waite, "Software Manual for the Elementary
//     Functions", 1980): k = nearest integer to phi * 2/pi (the product formed with
//     2/pi in two binary32 parts), r = phi - k * pi/2 with pi/2
//     split into three binary32 parts P1 + P2 + P3 (72 bits).  Each k * Pi is formed
//     exactly as a sum of two binary32 numbers with a fused multiply-add, phi - k*P1 is
//     exact (Sterbenz), and the rest is summed as a double-float (an unevaluated sum of
//     two binary32 numbers, Dekker 1971).  For phi < 2^24, k < 2^23.4 and the absolute
//     error of r stays below 2^-45.
//  2. sin r and cos r on |r| <= pi/4 from their Taylor series (coefficients (-1)^n / n!,
//     through r^15 and r^16), the leading terms in double-float arithmetic and the tail
//     in binary32 (Horner's rule); the truncation error is below 2^-54.
//  3. Quadrant: (cos phi, sin phi) = (cos r, sin r) rotated by k quarter turns.
//  4. Ziv's rounding test (Ziv 1991, "Fast evaluation of elementary mathematical
//     functions with correctly rounded last bit"): the double-float result y_h + y_l
//     is within eps of the exact value; if y_h's rounding interval contains
//     [y - eps, y + eps] with room to spare, y_h is RN32 of the exact value and of every
//     value within a few binary64 units of it -- so it equals the binary64 evaluation
//     rounded to binary32.  Otherwise the caller evaluates in binary64 as before: for
//     3.9e-5 of the angles in [2^-20, 2^24).
//
// eps = 2^-42 |y| + (k != 0 ? 2^-43 : 0).  Over every binary32 angle in [2^-20, 2^24)
// the double-float result is within 2^-44.9 |y| (relative) and, for k != 0, 2^-45.4
// (absolute) of the exact value, so eps holds with a factor of 5 or more to spare; the
// margin also covers the binary64 evaluation's own error (a few units of 2^-53
// relative) and its rounding to binary32.  Angles at or above 2^24, negative, NaN or
// infinite go to the binary64 path.  Angles below 2^-13 need no evaluation: cos phi
// rounds to 1 and sin phi to phi.  A test compares this with the binary64 evaluation
// on every binary32 angle in [2^-20, 2^24) and on samples of the rest.
#pragma once

#include <cstdint>

namespace pvr {

// A double-float: the unevaluated sum hi + lo, |lo| <= ulp(hi) / 2.
struct DF {
    float hi, lo;
};

// Exact sum a + b = s + e (Knuth's two-sum, no ordering assumption).
__device__ __forceinline__ DF two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// Exact sum a + b = s + e when |a| >= |b| or a == 0 (Dekker's fast two-sum).
__device__ __forceinline__ DF fast_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// Exact product a * b = p + e with one fused multiply-add.
__device__ __forceinline__ DF two_prod(float a, float b)
{
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

// Double-float products and sums (relative error a few units of 2^-48).
__device__ __forceinline__ DF df_mul(DF a, DF b)
{
    DF p = two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
    return fast_two_sum(p.hi, p.lo);
}

__device__ __forceinline__ DF df_mul_f(DF a, float b)
{
    DF p = two_prod(a.hi, b);
    p.lo = __fmaf_rn(a.lo, b, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

__device__ __forceinline__ DF df_add(DF a, DF b)
{
    DF s = two_sum(a.hi, b.hi);
    s.lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    return fast_two_sum(s.hi, s.lo);
}

// A binary64 constant as a double-float (its leading 48 bits).
struct DFConst {
    float hi, lo;
    __host__ __device__ constexpr DFConst(double v) : hi(static_cast<float>(v)), lo(static_cast<float>(v - static_cast<double>(static_cast<float>(v)))) {}
    __device__ __forceinline__ DF df() const { return {hi, lo}; }
};

// 1/n! for the series, as binary64 values computed from the factorials.
constexpr double kInvFact2 = 1.0 / 2.0;
constexpr double kInvFact3 = 1.0 / 6.0;
constexpr double kInvFact4 = 1.0 / 24.0;
constexpr double kInvFact5 = 1.0 / 120.0;
constexpr double kInvFact6 = 1.0 / 720.0;
constexpr double kInvFact7 = 1.0 / 5040.0;
constexpr double kInvFact8 = 1.0 / 40320.0;
constexpr double kInvFact9 = 1.0 / 362880.0;
constexpr double kInvFact10 = 1.0 / 3628800.0;
constexpr double kInvFact11 = 1.0 / 39916800.0;
constexpr double kInvFact12 = 1.0 / 479001600.0;
constexpr double kInvFact13 = 1.0 / 6227020800.0;
constexpr double kInvFact14 = 1.0 / 87178291200.0;
constexpr double kInvFact15 = 1.0 / 1307674368000.0;
constexpr double kInvFact16 = 1.0 / 20922789888000.0;

// pi/2 = P1 + P2 + P3 + (1.1e-23): P1 = RN32(pi/2), P2 = RN32(pi/2 - P1),
// P3 = RN32(pi/2 - P1 - P2) (checked against a 300-bit pi by tests/test_cos_sin_constants.py).
constexpr float kPio2_1 = 0x1.921fb6p+0f;
constexpr float kPio2_2 = -0x1.777a5cp-25f;
constexpr float kPio2_3 = -0x1.ee59dap-50f;
constexpr float kTwoOverPi_1 = 0x1.45f306p-1f;      // RN32(2/pi)
constexpr float kTwoOverPi_2 = 0x1.b93910p-26f;     // RN32(2/pi - kTwoOverPi_1)
constexpr float kFastLimit = 0x1p+24f;               // angles the reduction covers
constexpr float kTinyAngle = 0x1p-13f;              // below: cos -> 1, sin -> phi
constexpr float kEpsRel = 0x1p-42f;
constexpr float kEpsAbsReduced = 0x1p-43f;

// RN32 of the exact value y_h + y_l +- eps when that is certain: true and y_h.
__device__ __forceinline__ bool round_certain(DF y, float eps_abs, float &out)
{
    const float ay = fabsf(y.hi);
    if (!(ay >= 0x1p-60f)) return false;
    const uint32_t bits = __float_as_uint(ay);
    // half the gap to the neighbouring binary32 numbers: 2^(e-24), or 2^(e-25) below a
    // power of two
    float half_gap = __uint_as_float((bits & 0x7f800000u) - (24u << 23));
    if ((bits & 0x007fffffu) == 0) half_gap = __fmul_rn(half_gap, 0.5f);
    const float eps = __fmaf_rn(kEpsRel, ay, eps_abs);
    if (__fsub_rn(half_gap, fabsf(y.lo)) > eps) {
        out = y.hi;
        return true;
    }
    return false;
}

// (RN32(cos phi), RN32(sin phi)) when the binary32 evaluation decides them: returns true
// with the pair; false when the caller must evaluate in binary64.
__device__ __forceinline__ bool cos_sin_binary32(float phi, float &c_out, float &s_out)
{
    if (!(phi >= 0.0f && phi < kFastLimit)) return false;
    if (phi < kTinyAngle) {
        c_out = 1.0f;
        s_out = phi;
        return true;
    }
    // 1. k = the integer nearest phi * 2/pi.  The product is formed from a two-part 2/pi
    //    (its leading part exactly, with an FMA), because its binary32 rounding alone is
    //    a whole unit apart above 2^23 and would leave |r| well beyond pi/4; the
    //    fraction it leaves picks between k0 and its neighbours.
    const DF x = two_prod(phi, kTwoOverPi_1);
    const float x_lo = __fmaf_rn(phi, kTwoOverPi_2, x.lo);
    float kf = rintf(x.hi);
    const float frac = __fadd_rn(__fsub_rn(x.hi, kf), x_lo);   // x.hi - kf is exact
    if (frac > 0.5f) kf = __fadd_rn(kf, 1.0f);
    else if (frac < -0.5f) kf = __fsub_rn(kf, 1.0f);
    //    r = phi - k pi/2 as a double-float
    DF r;
    float eps_abs = 0.0f;
    if (kf == 0.0f) {
        r = {phi, 0.0f};
    } else {
        const DF p1 = two_prod(kf, kPio2_1);
        const DF p2 = two_prod(kf, kPio2_2);
        const float p3 = __fmul_rn(kf, kPio2_3);
        const float t = __fsub_rn(phi, p1.hi);                  // exact (Sterbenz)
        const DF a = two_sum(t, -p1.lo);
        const DF b = two_sum(a.hi, -p2.hi);
        const float tail = __fsub_rn(__fsub_rn(__fadd_rn(a.lo, b.lo), p2.lo), p3);
        r = two_sum(b.hi, tail);
        eps_abs = kEpsAbsReduced;
    }
    // 2. u = r^2; sin r = r + r u S(u), cos r = 1 - u/2 + u^2 C(u)
    const float uh0 = __fmul_rn(r.hi, r.hi);
    const float ul0 = __fmaf_rn(__fmul_rn(2.0f, r.hi), r.lo, __fmaf_rn(r.hi, r.hi, -uh0));
    const DF u = fast_two_sum(uh0, ul0);
    const float uh = u.hi;
    // binary32 tails (their terms are below 2^-21 of the result)
    const float s_tail = static_cast<float>(kInvFact9) +
                         uh * (-static_cast<float>(kInvFact11) +
                               uh * (static_cast<float>(kInvFact13) - uh * static_cast<float>(kInvFact15)));
    const float c_tail = static_cast<float>(kInvFact10) -
                         uh * (static_cast<float>(kInvFact12) -
                               uh * (static_cast<float>(kInvFact14) - uh * static_cast<float>(kInvFact16)));
    // double-float steps
    DF sp = df_add(DFConst(-kInvFact7).df(), df_mul_f(u, s_tail));
    sp = df_add(DFConst(kInvFact5).df(), df_mul(u, sp));
    sp = df_add(DFConst(-kInvFact3).df(), df_mul(u, sp));      // S(u)
    DF cp = df_add(DFConst(kInvFact8).df(), df_mul_f(u, -c_tail));
    cp = df_add(DFConst(-kInvFact6).df(), df_mul(u, cp));
    cp = df_add(DFConst(kInvFact4).df(), df_mul(u, cp));       // C(u)
    const DF ru = df_mul(r, u);
    const DF sin_r = df_add(r, df_mul(ru, sp));
    const DF u2 = df_mul(u, u);
    const DF minus_half_u = {__fmul_rn(-0.5f, u.hi), __fmul_rn(-0.5f, u.lo)};   // exact
    const DF cos_r = df_add(DF{1.0f, 0.0f}, df_add(minus_half_u, df_mul(u2, cp)));
    // 3. quadrant
    const int q = static_cast<int>(kf) & 3;
    DF cv = (q & 1) ? sin_r : cos_r;
    DF sv = (q & 1) ? cos_r : sin_r;
    if (q == 1 || q == 2) cv = {-cv.hi, -cv.lo};
    if (q == 2 || q == 3) sv = {-sv.hi, -sv.lo};
    // 4. rounding test
    return round_certain(cv, eps_abs, c_out) && round_certain(sv, eps_abs, s_out);
}

}  // namespace pvr
