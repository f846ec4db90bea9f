/*
 * Test and tuning entry points of libspecverify (not part of the verify path):
 * per-call options, introspection, and checks of the draw's arithmetic.
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

/* Options of one call, for tests and tuning.  Every field 0 means the
 * automatic choice (what the entry points of specverify.h always use).  They
 * apply to the one call they are passed to (the _tuned entry points below), so
 * a test or a tuning script never changes the behaviour of another caller of
 * the library.  A field outside its range makes the call return
 * SV_ERR_INVALID_ARG.
 *   path           1 the two-kernel path, 2 the fused per-sequence kernel, 3 the
 *                  row-skipping path (0 automatic: the row-skipping path when B
 *                  is at least the SM count, or in sampled mode half of it;
 *                  else, in sampled mode, the fused kernel when rows are at most
 *                  1 KiB or its clusters cover every SM; else the two-kernel
 *                  path);
 *   force_precise  1: every sampled draw takes the precise float-float pass;
 *   draw_split     the sampled draw kernel's cluster size (1, 2, 4, 8, 16); under
 *                  the split draw, at most this many slices per row;
 *   precise_split  the cluster size of the precise-draw kernel of large batches;
 *   fused_defer    the fused kernel hands the draws that need the precise pass
 *                  to a separate kernel: 1 always, 2 never (0: when B is at
 *                  least the SM count);
 *   fused_pad_kib  the fused kernel's minimum dynamic shared memory per CTA
 *                  (KiB, up to 160), limiting how many share an SM;
 *   rows_split     the row stream's CTAs per row (1..16, a power of two): a
 *                  cluster per row on the two-kernel path; on the row-skipping
 *                  path (at most 8; automatic: 1) separate CTAs merged through
 *                  the workspace;
 *   rows_threads   its threads per CTA (128, 256, 512 or 1024);
 *   flat_off       1: greedy batches never take the flat row stream (the whole
 *                  logits tensor cut into one equal range per resident CTA);
 *                  a fixed rows_split or rows_threads also keeps them off it;
 *   draw_mode      the sampled draw of the two-kernel and row-skipping paths:
 *                  1 the split draw (slices of the decision row on separate
 *                  CTAs, when the workspace holds its sums), 2 the cluster
 *                  draw (one cluster per sequence); 0 automatic (the split
 *                  draw when the workspace holds its sums, else the cluster
 *                  draw). */
typedef struct {
    int path;
    int force_precise;
    int draw_split;
    int precise_split;
    int fused_defer;
    int fused_pad_kib;
    int rows_split;
    int rows_threads;
    int flat_off;
    int draw_mode;
} sv_tuning;

/* spec_verify_sample / spec_verify_sample_kv (kv_len and stats may be NULL),
 * spec_verify_greedy / spec_verify_greedy_kv, spec_verify_rows,
 * spec_verify_finish, spec_verify_tree and spec_verify_match with the options
 * of `tuning` (NULL: the automatic choices).  Arguments, results and errors
 * otherwise as for those calls. */
sv_status spec_verify_sample_tuned(const void* logits, sv_dtype dtype, const float* draft_probs,
                                   const int32_t* draft_tokens, const float* u_accept,
                                   const float* u_resample, float T, int B, int k, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                   cudaStream_t stream, const sv_tuning* tuning);
sv_status spec_verify_greedy_tuned(const void* logits, sv_dtype dtype,
                                   const int32_t* draft_tokens, int B, int k, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                   cudaStream_t stream, const sv_tuning* tuning);
sv_status spec_verify_rows_tuned(sv_mode mode, const void* logits, sv_dtype dtype,
                                 const float* draft_probs, const int32_t* draft_tokens, float T,
                                 int B, int k, int V, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, const sv_tuning* tuning);
sv_status spec_verify_finish_tuned(sv_mode mode, const void* logits, sv_dtype dtype,
                                   const float* draft_probs, const int32_t* draft_tokens,
                                   const float* u_accept, const float* u_resample, float T,
                                   int B, int k, int V, int32_t* out_tokens,
                                   int32_t* num_accepted, void* ws, size_t ws_bytes,
                                   cudaStream_t stream, const sv_tuning* tuning);
sv_status spec_verify_tree_tuned(sv_mode mode, const void* logits, sv_dtype dtype,
                                 const float* draft_probs, const int32_t* tree_tokens,
                                 const int32_t* tree_parents, const float* u_accept,
                                 const float* u_resample, float T, int B, int N, int V,
                                 int32_t* out_tokens, int32_t* out_nodes, int32_t* num_accepted,
                                 void* ws, size_t ws_bytes, cudaStream_t stream,
                                 const sv_tuning* tuning);
sv_status spec_verify_match_tuned(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                                  const float* u_draw, const float* u_bonus, float T, int B, int k,
                                  int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                  size_t ws_bytes, cudaStream_t stream, const sv_tuning* tuning);

/* The path (1, 2 or 3 as above) the one-call entry points of specverify.h
 * take for these sizes on the current device, -1 on error or bad sizes. */
int spec_verify_debug_path(sv_mode mode, int B, int V, sv_dtype dtype);

/* The number of CTAs of the flat greedy row stream that spec_verify_greedy (or
 * spec_verify_rows in greedy mode) launches for these sizes on the current
 * device with 16-byte aligned logits; 0 when it takes the per-row stream;
 * -1 on error or bad sizes. */
int spec_verify_debug_flat_ctas(int B, int k, int V, sv_dtype dtype);

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

/* Synchronises `stream`; counts[i] receives the number of sequences of the
 * last call on `ws` whose status word has bit i set (bit 5, SV_DEV_PRECISE:
 * the draws that needed the float-float pass).  HOST array of 8. */
sv_status spec_verify_debug_status_counts(const void* ws, cudaStream_t stream,
                                          uint32_t counts[8]);

/* Writes to *out (a DEVICE float) the largest relative error of the
 * ex2.approx.ftz.f32 instruction against the float-float 2^a over every float a
 * in [a0, a1], -126 <= a0 <= a1 <= 0.  The fast draw's error bound assumes this
 * is at most 1.75e-7 over [-126, 0] (a test checks it exhaustively).
 * Synchronises `stream`.  SV_ERR_INVALID_ARG for a bad range or a null pointer. */
sv_status spec_verify_debug_ex2_error(float a0, float a1, float* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
