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

#ifdef __cplusplus
}
#endif
#endif
