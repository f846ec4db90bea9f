// Float-float ("double-single") arithmetic for the high-precision draw.
//
// A value is an unevaluated sum hi + lo of two floats carrying about 48
// significant bits.  The error-free transformations are the classical ones:
// TwoSum (Knuth, TAOCP vol. 2, 4.2.2), Fast2Sum (Dekker 1971, valid when
// |a| >= |b|) and the FMA-based exact product.  Every operation uses the
// explicitly rounded intrinsics (__fadd_rn, __fmul_rn, __fmaf_rn) so that no
// compiler contraction can change a rounding these transformations rely on.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

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

// Sum of two float-float values, renormalised; accurate to ~2^-47 relative when
// both operands have the same sign (all sums in this library are of
// non-negative terms).
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    ff s = two_sum(a.hi, b.hi);
    float lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    return fast_two_sum(s.hi, lo);
}

// Running sum of non-negative float-float terms: the high parts are added with
// an exact TwoSum whose error, with the low parts, collects in `lo` without
// renormalisation.  Each TwoSum error is at most 2^-24 of the running `hi`, so
// after n terms |lo| <= n 2^-24 hi, and the float additions into `lo` add at
// most n^2 2^-48 hi of their own: about 2^-31 of hi for the few hundred terms
// one thread sums in this library (2^-42 for a chunk of 8).
__device__ __forceinline__ void ff_accumulate(ff& acc, ff t) {
    ff s = two_sum(acc.hi, t.hi);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(acc.lo, __fadd_rn(s.lo, t.lo));
}

__device__ __forceinline__ ff ff_normalize(ff a) { return fast_two_sum(a.hi, a.lo); }

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
    float res = __fmaf_rn(-s.hi, r, 1.0f);  // 1 - s.hi * r, exact up to one rounding
    res = __fmaf_rn(-s.lo, r, res);         // - s.lo * r
    return fast_two_sum(r, __fmul_rn(res, r));
}

// ------------------------------------------------------------------ 2^(i/1024) table
//
// Built at compile time: 2^(i/1024) = exp(i ln2 / 1024) summed as its Taylor
// series in double precision (30 terms for arguments below ln 2, truncation far
// below 2^-53), then split into float-float.  ln 2 enters as its decimal value.
constexpr double kLn2 = 0.693147180559945309417232121458176568;

constexpr double exp_series(double x) {
    double term = 1.0, sum = 1.0;
    for (int n = 1; n < 30; ++n) {
        term = term * x / n;
        sum = sum + term;
    }
    return sum;
}

constexpr int kExpTableBits = 10;
constexpr int kExpTable = 1 << kExpTableBits;

struct Exp2Table {
    float hi[kExpTable];
    float lo[kExpTable];
};

constexpr Exp2Table make_exp2_table() {
    Exp2Table t{};
    for (int i = 0; i < kExpTable; ++i) {
        double v = exp_series((double)i * kLn2 / kExpTable);
        t.hi[i] = (float)v;
        t.lo[i] = (float)(v - (double)t.hi[i]);
    }
    return t;
}

// Lower end of the exponent range evaluated: 2^-66 is below the 2^-60
// resolution of the fixed-point weights even for the largest normaliser.
constexpr float kExp2Min = -66.0f;

// 2^a for a float-float a = (ah, al) with kExp2Min <= ah <= 0 (al tiny), to
// ~2^-45 relative.  a = K/1024 + r with an integer K and |r| <= 2^-11;
// 2^a = 2^(K div 1024) * T[K mod 1024] * exp(r ln2), T from the table and
// exp(s), |s| <= 3.4e-4, from its Taylor series to s^4 (next term < 6e-17):
// s and 1 in float-float, the higher terms in float.
__device__ __forceinline__ ff exp2_ff(float ah, float al, const float* __restrict__ thi,
                                      const float* __restrict__ tlo) {
    const float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer
    float t = __fmaf_rn(ah, (float)kExpTable, kMagic);
    float kf = __fsub_rn(t, kMagic);
    int ki = __float_as_int(t) - 0x4B400000;
    float r1 = __fmaf_rn(kf, -1.0f / kExpTable, ah);  // exact (Sterbenz)
    // The reduced argument r = r1 + al, renormalised: al can be a few percent of
    // r1, and the polynomial below uses the leading part alone.
    const ff r = two_sum(r1, al);
    // s = r * ln2 as a float-float pair (sh, sl).
    const float l2h = (float)kLn2;
    const float l2l = (float)(kLn2 - (double)(float)kLn2);
    float sh = __fmul_rn(r.hi, l2h);
    float sl = __fmaf_rn(r.hi, l2h, -sh);
    sl = __fmaf_rn(r.hi, l2l, sl);
    sl = __fmaf_rn(r.lo, l2h, sl);
    // exp(s) - 1 - sh = sl + s^2/2 + s^3/6 + s^4/24 (+ the sh*sl cross term)
    float c = __fmaf_rn(sh, 1.0f / 24.0f, 1.0f / 6.0f);
    c = __fmaf_rn(sh, c, 0.5f);
    float tail = __fmaf_rn(__fmul_rn(sh, sh), c, __fmaf_rn(sh, sl, sl));
    ff e1 = fast_two_sum(1.0f, sh);
    e1.lo = __fadd_rn(e1.lo, tail);
    const int idx = ki & (kExpTable - 1);
    ff tb = {thi[idx], tlo[idx]};
    float ph = __fmul_rn(tb.hi, e1.hi);
    float pl = __fmaf_rn(tb.hi, e1.hi, -ph);
    pl = __fmaf_rn(tb.hi, e1.lo, pl);
    pl = __fmaf_rn(tb.lo, e1.hi, pl);
    const int j = ki >> kExpTableBits;  // floor(K / 1024) >= -66: 2^j is a normal float
    const float sc = __int_as_float((j + 127) << 23);
    return ff{__fmul_rn(ph, sc), __fmul_rn(pl, sc)};
}

// e = exp((l - m)/T) = 2^((l - m) * log2(e)/T) for l <= m, with c = log2(e)/T
// as float-float; 0 when the exponent is below kExp2Min (and for l = -inf).
// Branch-free: out-of-range arguments are evaluated at 0 and the result masked,
// so the lanes of a warp never diverge here.
__device__ __forceinline__ ff exp_rel(float l, float m, ff c, const float* __restrict__ thi,
                                      const float* __restrict__ tlo) {
    ff d = two_sum(l, -m);  // l - m exactly
    float ah = __fmul_rn(d.hi, c.hi);
    float al = __fmaf_rn(d.hi, c.hi, -ah);
    al = __fmaf_rn(d.hi, c.lo, al);
    al = __fmaf_rn(d.lo, c.hi, al);
    const bool ok = ah >= kExp2Min;  // false for NaN and -inf too
    ff e = exp2_ff(ok ? ah : 0.0f, ok ? al : 0.0f, thi, tlo);
    return ff{ok ? e.hi : 0.0f, ok ? e.lo : 0.0f};
}

// ------------------------------------------------------------------ fixed point
//
// Weights become unsigned 64-bit integers in units of 2^-60 so that prefix sums
// are exact and independent of summation order.  The conversion uses only
// integer operations on the float's bits (no int64 conversion instruction).

constexpr int kFixBits = 60;

// round-toward-zero of |x| * 2^60 for |x| < 16, branch-free.
__device__ __forceinline__ unsigned long long fix_mag(float x) {
    const uint32_t b = __float_as_uint(x) & 0x7FFFFFFFu;
    const int ex = (int)(b >> 23);
    const unsigned long long mant = (unsigned long long)((b & 0x7FFFFFu) | 0x800000u);
    const int sh = ex - 127 - 23 + kFixBits;  // <= 40 for |x| < 16
    const unsigned long long left = mant << (sh > 0 ? sh : 0);
    const unsigned long long right = mant >> (sh < 0 ? (sh > -63 ? -sh : 63) : 0);
    const unsigned long long v = sh >= 0 ? left : right;
    return ex == 0 ? 0ull : v;  // zero or subnormal: below the resolution
}

// floor(x 2^s) for a float x >= 0 and 0 <= s <= 127 with x 2^s < 2^64.  The
// scaled value v = x 2^s is exact, and so are its two halves: h = floor(v /
// 2^32) has at most 24 significant bits (v has 24), and v - h 2^32, a multiple
// of ulp(v) below 2^32, fits a float too; each half is converted toward zero
// (32-bit conversions: a 64-bit one runs on the narrow FP64 pipe).  Zero and
// subnormal x give 0 (x 2^s < 2^-3 then).
__device__ __forceinline__ unsigned long long fix_pow2(float x, int s) {
    const float v = __fmul_rn(x, __int_as_float((127 + s) << 23));
    const float hf = __fmul_rn(v, 2.3283064365386963e-10f);  // v / 2^32
    const uint32_t h = __float2uint_rz(hf);
    const float lf = __fmaf_rn(-__uint2float_rn(h), 4294967296.0f, v);
    const uint32_t l = __float2uint_rz(lf);
    return ((unsigned long long)h << 32) | l;
}

// Fixed-point value of a non-negative float-float (hi >= 0, |lo| <= ulp(hi)).
__device__ __forceinline__ unsigned long long to_fixed(ff v) {
    unsigned long long h = fix_mag(v.hi);
    unsigned long long l = fix_mag(v.lo);
    return v.lo < 0.0f ? h - l : h + l;
}

}  // namespace sv
