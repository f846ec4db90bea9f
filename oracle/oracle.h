/*
 * Plain float64 CPU oracle for the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm use it.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   [DEE] "Decodificação especulativa explicada: rascunhe barato, verifique numa
 *         passada" (gsantana.dev)
 *   [SD15] "Speculative Decoding", ch15 of "LLM serving from scratch"
 *         (snowch.github.io)
 *   [SDF] "Speculative decoding: el secretario que adelanta lo que va a decir el
 *         jefe — fundamentos, matemáticas y estado mayo 2026" (blog.lo0.es)
 */
#ifndef SV_ORACLE_H
#define SV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Verify modes. */
enum {
    ORC_SAMPLE = 0,       /* rejection sampling, [DEE] §"A regra de amostragem por rejeição" */
    ORC_GREEDY = 1,       /* accept while draft == argmax, [DEE] same section, last paragraph */
    ORC_SAMPLE_BUGGY = 2, /* negative control: resample from p instead of the residual,
                             [DEE] §"A regra de amostragem por rejeição" (the "Júnior" aside),
                             [SD15] §"Why the result is exactly the target model" */
    ORC_MATCH = 3         /* sample-and-match: draw a target token at every position and keep
                             the draft's while they agree, [DEE] §"A regra de amostragem por
                             rejeição", the simpler exact scheme; the draw at position i < k
                             uses ua[i], the one at position k uses ur; q is not used */
};

/* Per-sequence flag bits written by the oracle. */
enum {
    ORC_F_BAD = 1,         /* a row / token / uniform the scan needed was invalid */
    ORC_F_DEGENERATE = 2,  /* rejected but the residual had zero mass: drew from p instead */
    ORC_F_OVERFLOW = 4     /* the draw ran past the last bin: clamped to the last positive bin */
};

/* Row statistics of one logits row (float64 input).
 * m = max_j l_j / T, S = sum_j exp(l_j/T - m) (Neumaier-compensated),
 * argmax = lowest j holding the largest raw l_j.
 * Returns 1 if the row is invalid (a NaN, a +inf, or every entry -inf), else 0. */
int orc_row_stats(const double* l, double T, int V, double* m, double* S, int32_t* argmax);

/* Normalised cumulative boundaries cdf[j] = C_j / C_{V-1} of the weights the draw
 * uses for one row: w_j = max(0, p_j - q_j) when q != NULL, else w_j = p_j.
 * Returns 0, or 1 when the total weight is zero (cdf left untouched). */
int orc_draw_cdf(const double* l, const double* q, double T, int V, double* cdf);

/* One sequence, all inputs already float64.
 *   logits [k+1][V], q [k][V] (unused in greedy), x [k], ua [k] (unused in greedy),
 *   ur (unused in greedy), T > 0 (greedy ignores it).
 * Outputs: out [k+1] (drafts 0..n-1, the drawn token at n, -1 after),
 *   *n_acc = n in [0,k] (-1 if the sequence is invalid),
 *   thr [k] (may be NULL): min(1, P/Q) at every judged sampled position, NaN elsewhere,
 *   *draw_lo / *draw_hi (may be NULL): C_{t-1}/C_tot and C_t/C_tot of the drawn bin
 *   (NaN in greedy mode), *flags (may be NULL): ORC_F_* bits. */
void orc_verify_seq(int mode, const double* logits, const double* q, const int32_t* x,
                    const double* ua, double ur, double T, int k, int V,
                    int32_t* out, int32_t* n_acc, double* thr, double* draw_lo,
                    double* draw_hi, int32_t* flags);

/* Batch form over B independent sequences, inputs in the device layouts:
 *   logits [B][k+1][V] as bf16 bit patterns (dtype 0, uint16) or float32 (dtype 1),
 *   q [B][k][V] float32, x [B][k] int32, ua [B][k] float32, ur [B] float32.
 * Every per-row / per-sequence output pointer may be NULL.
 *   row_m, row_S, row_px, row_qx: [B][k+1] float64 (px, qx are NaN on row k and for
 *   out-of-range draft tokens); row_argmax [B][k+1]; thr [B][k];
 *   draw_lo, draw_hi, flags [B].
 * nthreads <= 0 uses the OpenMP default.  Returns 0, or -1 on bad arguments. */
int orc_verify_batch(int mode, const void* logits, int dtype, const float* q,
                     const int32_t* x, const float* ua, const float* ur, float T,
                     int B, int k, int V, int32_t* out, int32_t* n_acc,
                     double* row_m, double* row_S, int32_t* row_argmax,
                     double* row_px, double* row_qx, double* thr,
                     double* draw_lo, double* draw_hi, int32_t* flags, int nthreads);

/* Step 1 over R rows in the device layout (bf16 bit patterns, dtype 0, or
 * float32, dtype 1), R = B*(k+1) for a batch: m[r], S[r], argmax[r] as
 * orc_row_stats gives them at temperature T, bad[r] its return value. */
int orc_row_stats_batch(const void* logits, int dtype, float T, int R, int V, double* m,
                        double* S, int32_t* argmax, int32_t* bad, int nthreads);

/* orc_verify_batch for modes ORC_SAMPLE, ORC_GREEDY and ORC_SAMPLE_BUGGY with
 * the per-row statistics supplied instead of recomputed: st_m, st_S,
 * st_argmax, st_bad [B][k+1] as orc_row_stats_batch returned them for these
 * logits (at T, or at 1 in greedy mode).  Wherever the scan or the draw needs a
 * row's statistics it reads them there; every other step, and every output,
 * is that of orc_verify_batch (which has no per-row outputs here).  For
 * verifying one set of logits many times with fresh drafts and uniforms. */
int orc_verify_batch_stats(int mode, const void* logits, int dtype, const float* q,
                           const int32_t* x, const float* ua, const float* ur, float T, int B,
                           int k, int V, const double* st_m, const double* st_S,
                           const int32_t* st_argmax, const int32_t* st_bad, int32_t* out,
                           int32_t* n_acc, double* thr, double* draw_lo, double* draw_hi,
                           int32_t* flags, int nthreads);

/* Number of OpenMP threads a batch call with nthreads <= 0 would use. */
int orc_max_threads(void);

/* N-gram (prompt-lookup) drafter ([DEE] §"A família de rascunhos", prompt
 * lookup: find the last tokens earlier in the context and propose what
 * followed them there; [SD15] §"What proposes the tokens", NgramDrafter).  For
 * each sequence b with history h = history[b*Lmax .. b*Lmax + lengths[b]):
 * for n = n_max down to n_min, look for earlier occurrences of the last n
 * tokens, h[e-n+1 .. e] == h[L-n .. L-1] with e <= L-2; the first n with an
 * occurrence wins, and of its occurrences the most recent (largest e).  The
 * draft is h[e+1 .. e+k], cut at the end of the history: num[b] tokens, -1
 * after.  No occurrence (or L < n_min + 1): num[b] = 0.  Returns 0, or -1 for
 * bad arguments. */
int orc_ngram_draft(const int32_t* history, const int32_t* lengths, int B, int Lmax, int k,
                    int n_min, int n_max, int32_t* draft, int32_t* num);

/* Tree verification of several candidates at once ([DEE] §"A família de
 * rascunhos", Medusa: extra heads propose several continuations that the
 * target checks in one pass with tree attention; [SDF] §"Tree attention": how
 * Medusa and EAGLE-2 verify several candidates).  The pages give the idea, not
 * a rule; this is the plainest exact reading, which reduces to the chain rule
 * when every node has one child.
 *
 * One sequence's tree of N nodes: node 0 is the root (the last committed
 * token); node j >= 1 carries the drafted token tok[j] and its parent par[j],
 * 0 <= par[j] < j.  logits [N][V]: the target's logits at each node (the
 * distribution of the token after it).  q [N][V] (sampled): the draft
 * distribution at each node, from which its children were drawn independently.
 * ua [N]: the uniform of the test of child j (ua[0] unused); ur: the final draw.
 *
 * The walk starts at the root.  Greedy: the first child (in index order) whose
 * token is the argmax of the current node is accepted and the walk moves to
 * it; when none is, the argmax is emitted.  Sampled (recursive rejection over
 * the children): the current distribution r starts as p = softmax(l/T) of the
 * node; each child j in index order is accepted iff r(x) >= q(x) or
 * ua[j] < r(x)/q(x), x = tok[j], q the node's draft distribution; on
 * rejection r becomes the normalised residual max(0, r - q) (or p again, with
 * ORC_F_DEGENERATE, when that has no mass).  After an acceptance the walk
 * moves to the child with r = its own p; when no child is accepted the final
 * token is drawn from r (step 4's rule on the unnormalised residual weights)
 * with ur.  Each tested child contributes thr[j] = min(1, r(x)/q(x)).
 *
 * Mode ORC_SAMPLE_BUGGY (a negative control for the tests): each sibling is
 * tested against p itself and the final draw uses the residual of p taken once,
 * as if each sibling were a fresh chain step; this does not preserve p.
 * Outputs: out [N] (the accepted tokens, the emitted token, -1 after),
 * nodes [N] (the accepted node indices, -1 after), *n_acc (-1 if invalid:
 * a bad parent anywhere, or a row, token, uniform or q(x) the walk needs),
 * thr [N] (NaN for untested nodes), draw_lo / draw_hi, flags. */
void orc_tree_seq(int mode, const double* logits, const double* q, const int32_t* tok,
                  const int32_t* par, const double* ua, double ur, double T, int N, int V,
                  int32_t* out, int32_t* nodes, int32_t* n_acc, double* thr, double* draw_lo,
                  double* draw_hi, int32_t* flags);

/* Batch form: logits [B][N][V] (bf16 bit patterns, dtype 0, or float32,
 * dtype 1), q [B][N][V] float32, tok / par [B][N] int32, ua [B][N] float32,
 * ur [B] float32; out / nodes [B][N], n_acc [B]; row_m, row_argmax [B][N] and
 * thr [B][N], draw_lo, draw_hi, flags [B] may be NULL.  Returns 0, or -1 on
 * bad arguments. */
int orc_tree_batch(int mode, const void* logits, int dtype, const float* q, const int32_t* tok,
                   const int32_t* par, const float* ua, const float* ur, float T, int B, int N,
                   int V, int32_t* out, int32_t* nodes, int32_t* n_acc, double* row_m,
                   int32_t* row_argmax, double* thr, double* draw_lo, double* draw_hi,
                   int32_t* flags, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
