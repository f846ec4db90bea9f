// Float-float ("double-single") arithmetic for the high-precision draw.
//
// A value is an unevaluated sum hi + lo of two floats with |lo| <= ulp(hi)/2,
// carrying about 48 significant bits.  The error-free transformations are the
// classical ones: TwoSum (Knuth, TAOCP vol. 2, 4.2.2), Fast2Sum (Dekker 1971,
// valid when |a| >= |b|) and the FMA-based exact product.  Every operation uses
// the explicitly rounded intrinsics (__fadd_rn, __fmul_rn, __fmaf_rn) so that no
// compiler contraction can change a rounding these transformations rely on.
#pragma once

#include <cuda_runtime.h>

namespace sv {

struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b) {
    float s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// Requires |a| >= |b| (or a == 0).
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
    float s = __fadd_rn(a, b);
    float e = __fsub_rn(b, __fsub_rn(s, a));
    return {s, e};
}

// Sum of two float-float values; the result is accurate to ~2^-47 relative
// when both operands have the same sign (all sums in this library are of
// non-negative terms).
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    ff s = two_sum(a.hi, b.hi);
    float lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    return fast_two_sum(s.hi, lo);
}

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
    float p = __fmul_rn(a.hi, b.hi);
    float e = __fmaf_rn(a.hi, b.hi, -p);
    e = __fmaf_rn(a.hi, b.lo, e);
    e = __fmaf_rn(a.lo, b.hi, e);
    return fast_two_sum(p, e);
}

// 1 / s for s > 0: the correctly rounded float reciprocal refined by one Newton
// step carried in float-float.
__device__ __forceinline__ ff ff_recip(ff s) {
    float r = __frcp_rn(s.hi);
    float res = __fmaf_rn(-s.hi, r, 1.0f);   // 1 - s.hi * r, exact up to one rounding
    res = __fmaf_rn(-s.lo, r, res);          // - s.lo * r
    return fast_two_sum(r, __fmul_rn(res, r));
}

// Constants of the exponential, computed on the host in double precision and
// passed to the kernels by value (see FFExpConst in the host code).
struct FFExpConst {
    float tbl_hi[64];  // 2^(i/64) split into float-float
    float tbl_lo[64];
    float c1, c2, c3;  // ln2/64 = c1 + c2 + c3, c1 with 12 significant bits
    float inv_l;       // 64 / ln2
};

// exp(y) for a float-float y <= 0 with y.hi >= -44, to ~2^-46 relative.
//
// Method: Tang's table-driven exponential (P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989) carried in float-float.  y = K ln2/64 + r
// with an integer K and |r| <= ln2/128; the reduction subtracts K*ln2/64 in the
// three pieces of Cody and Waite (the first, 12 bits long, makes K*c1 exact for
// |K| < 4096); exp(y) = 2^(K div 64) * 2^((K mod 64)/64) * exp(r), the middle
// factor from the 64-entry table and exp(r) from its Taylor series to r^5
// (the next term is below 4e-17): the r and r^2/2 terms in float-float, the
// cubic tail in float.
__device__ __forceinline__ ff ff_exp_neg(ff y, const float* __restrict__ thi,
                                         const float* __restrict__ tlo, float c1, float c2,
                                         float c3, float inv_l) {
    const float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer
    float t = __fmaf_rn(y.hi, inv_l, kMagic);
    float kf = __fsub_rn(t, kMagic);
    int ki = __float_as_int(t) - 0x4B400000;
    float r1 = __fmaf_rn(-kf, c1, y.hi);     // exact: K*c1 is exact, Sterbenz for the rest
    float p2 = __fmul_rn(kf, c2);
    float e2 = __fmaf_rn(kf, c2, -p2);       // exact error of K*c2
    ff s = two_sum(r1, -p2);
    float lo = __fadd_rn(__fsub_rn(__fsub_rn(s.lo, e2), __fmul_rn(kf, c3)), y.lo);
    ff r = fast_two_sum(s.hi, lo);

    float sq = __fmul_rn(r.hi, r.hi);
    float sqe = __fmaf_rn(r.hi, r.hi, -sq);
    float a = __fmaf_rn(r.hi, 1.0f / 120.0f, 1.0f / 24.0f);
    a = __fmaf_rn(r.hi, a, 1.0f / 6.0f);
    float cub = __fmul_rn(a, __fmul_rn(sq, r.hi));  // r^3/6 + r^4/24 + r^5/120
    float small = __fadd_rn(r.lo, __fmaf_rn(r.hi, r.lo, __fmaf_rn(sqe, 0.5f, cub)));
    ff em1 = fast_two_sum(r.hi, __fmul_rn(sq, 0.5f));   // r + r^2/2 (leading parts)
    float em1lo = __fadd_rn(em1.lo, small);
    ff b = fast_two_sum(1.0f, em1.hi);                  // exp(r) = 1 + expm1(r)
    b.lo = __fadd_rn(b.lo, em1lo);

    int idx = ki & 63;
    ff tb = {thi[idx], tlo[idx]};
    ff e = ff_mul(tb, b);
    int j = ki >> 6;  // floor(K / 64); j >= -64 here, so 2^j is a normal float
    float sc = __int_as_float((j + 127) << 23);
    e.hi = __fmul_rn(e.hi, sc);
    e.lo = __fmul_rn(e.lo, sc);
    return e;
}

}  // namespace sv
