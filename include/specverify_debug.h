/*
 * Test hooks of libspecverify (not part of the verify path).
 */
#ifndef SPECVERIFY_DEBUG_H
#define SPECVERIFY_DEBUG_H

#include "specverify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[i] = exp((l[i] - m) / T) evaluated by the float-float exponential of the
 * sampled draw (Tang's table-driven method carried in float-float), returned as
 * the double hi + lo; 0 where (l[i] - m)/T < -44.  l and out are DEVICE arrays
 * of n entries, l[i] <= m expected.  Asynchronous on `stream`.  Returns
 * SV_ERR_INVALID_ARG for a null pointer, n < 0 or T <= 0. */
sv_status spec_verify_debug_ffexp(const float* l, float m, float T, int n, double* out,
                                  cudaStream_t stream);

/* Route every sampled draw through the precise float-float pass (on != 0), or
 * back to the certified fast pass with fallback (on == 0, the default).  A
 * process-wide setting read at launch time, for tests only. */
void spec_verify_debug_force_precise(int on);

/* Choose the path of spec_verify_greedy / spec_verify_sample: 0 automatic
 * (the default: the fused per-sequence kernel when B is at least the SM count,
 * else the two-kernel path), 1 always the two-kernel path, 2 always the fused
 * kernel.  A process-wide setting read at launch time, for tests. */
void spec_verify_debug_force_path(int path);

/* 1 if the one-call entry points would run the fused kernel for a batch of B
 * sequences on the current device, 0 for the two-kernel path, -1 on error. */
int spec_verify_debug_uses_fused(int B);

/* Writes to *out (a DEVICE float) the largest relative error of the
 * ex2.approx.ftz.f32 instruction against the float-float 2^a over every float a
 * in [a0, a1], -126 <= a0 <= a1 <= 0.  The fast draw's error bound assumes this
 * is below 2^-21.  Synchronises `stream`.  SV_ERR_INVALID_ARG for a bad range
 * or a null pointer. */
sv_status spec_verify_debug_ex2_error(float a0, float a1, float* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
