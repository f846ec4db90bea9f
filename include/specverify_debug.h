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
 * (the default: the row-skipping path when B is at least the SM count, or in
 * sampled mode half of it; else, in sampled mode, the fused per-sequence kernel
 * when rows are at most 1 KiB or its clusters cover every SM; else the
 * two-kernel path), 1 always the two-kernel path, 2 always the
 * fused per-sequence kernel, 3 always the row-skipping path.  A process-wide
 * setting read at launch time, for tests. */
void spec_verify_debug_force_path(int path);

/* The path (1, 2 or 3 as above) the one-call entry points would take for these
 * sizes on the current device, -1 on error or bad sizes. */
int spec_verify_debug_path(sv_mode mode, int B, int V, sv_dtype dtype);

/* The number of CTAs of the flat greedy row stream that spec_verify_greedy (or
 * spec_verify_rows in greedy mode) would launch for these sizes on the current
 * device with 16-byte aligned logits; 0 when it would take the per-row stream;
 * -1 on error or bad sizes. */
int spec_verify_debug_flat_ctas(int B, int k, int V, sv_dtype dtype);

/* Fix the cluster size of the sampled draw kernel (spec_verify_finish and the
 * two-stage paths' second kernel) to G in {1, 2, 4, 8, 16}; 0 restores the
 * automatic choice; other values are ignored.  A process-wide setting read at
 * launch time, for tuning and tests. */
void spec_verify_debug_draw_split(int G);

/* Tuning of the fused per-sequence kernel: defer_mode 0 (default) hands the
 * draws that need the precise pass to a separate kernel when B is at least the
 * SM count, 1 always, 2 never; pad_kib > 0 gives every CTA at least that much
 * dynamic shared memory (KiB, up to 160), limiting how many share an SM.  Out
 * of range values are ignored.  A process-wide setting read at launch time. */
void spec_verify_debug_fused_tuning(int defer_mode, int pad_kib);

/* Fix the row stream's vocabulary split G (1, 2, 4, 8 or 16 CTAs per row) and
 * threads per CTA (128, 256 or 512) on the two-kernel path; 0 restores the
 * automatic choice of either; other values are ignored.  A process-wide setting
 * read at launch time, for tuning. */
void spec_verify_debug_rows_split(int G, int nt);

/* off = 1: greedy batches never take the flat row stream (the whole logits
 * tensor cut into one equal range per resident CTA, with per-row partial keys
 * merged by the finish kernel); they take the per-row stream instead.  0
 * restores the automatic choice.  A fixed split set with
 * spec_verify_debug_rows_split also turns the flat stream off.  For tests. */
void spec_verify_debug_flat(int off);

/* Fix the cluster size of the precise-draw kernel of large batches to G in
 * {1, 2, 4, 8, 16}; 0 restores the default.  For tuning. */
void spec_verify_debug_precise_split(int G);

/* The first stage of the row-skipping path alone: resets the per-sequence stop
 * rows in `ws` and runs the position-major row stream, leaving the row records
 * that spec_verify_finish reads (as spec_verify_rows does for the two-kernel
 * path; rows past a sequence's first stop may be left unread).  Arguments as
 * for spec_verify_rows, plus u_accept [B, k] fp32 (sampled mode, DEVICE).  For
 * timing the stages separately. */
sv_status spec_verify_debug_rows_skip(sv_mode mode, const void* logits, sv_dtype dtype,
                                      const float* draft_probs, const int32_t* draft_tokens,
                                      const float* u_accept, float T, int B, int k, int V,
                                      void* ws, size_t ws_bytes, cudaStream_t stream);

/* Writes to *out (a DEVICE float) the largest relative error of the
 * ex2.approx.ftz.f32 instruction against the float-float 2^a over every float a
 * in [a0, a1], -126 <= a0 <= a1 <= 0.  The fast draw's error bound assumes this
 * is at most 2^-22 over [-126, 0] (a test checks it exhaustively).  Synchronises `stream`.  SV_ERR_INVALID_ARG for a bad range
 * or a null pointer. */
sv_status spec_verify_debug_ex2_error(float a0, float a1, float* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
