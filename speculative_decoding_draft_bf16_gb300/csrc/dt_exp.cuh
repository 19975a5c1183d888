// Exponential and fixed-point masses of the acceptance walk.
#pragma once

#include "dt_device.cuh"

// ---------------------------------------------------------------------------
// exp_canon: fp32 exponential by Cody and Waite's argument reduction (W. J.
// Cody, W. Waite, "Software Manual for the Elementary Functions", 1980) and
// the Taylor series of e^r to degree 7 in Horner form.  Each step is one
// correctly rounded fp32 operation (explicit _rn intrinsics, no contraction),
// so the result is reproducible bit for bit on any IEEE machine with a fused
// multiply-add.  x < -86 gives 0, x > 88.5 gives +inf; every x <= 88.5 gives a
// finite value (e^88.5 < FLT_MAX).  Near the top k reaches 128, whose 2^k is
// not a float: it is applied as 2^127 * 2 (two exact scalings, one rounding).
// ---------------------------------------------------------------------------
DT_DI float dt_exp_canon(float x) {
    if (x != x) return x;
    if (x > 88.5f) return __int_as_float(0x7F800000);
    if (x < -86.0f) return 0.0f;
    const float log2e = 1.44269504088896340736f;
    const float c_hi = 0.693145751953125f;          // ln 2 rounded to 16 bits
    const float c_lo = 1.42860682030941723212e-6f;  // ln 2 - c_hi
    float kf = rintf(__fmul_rn(x, log2e));
    int k = (int)kf;
    float r = __fmaf_rn(-kf, c_hi, x);
    r = __fmaf_rn(-kf, c_lo, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    if (k > 127) return __fmul_rn(__fmul_rn(p, __int_as_float(254 << 23)), 2.0f);
    return __fmul_rn(p, __int_as_float((k + 127) << 23));
}

// floor(p * 2^32) for p in [0, 1] (exact scaling, then truncation).
DT_DI uint64_t dt_fixed32(float p) { return (uint64_t)__fmul_rn(p, 4294967296.0f); }

