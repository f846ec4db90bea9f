/*
 * Plain float64 CPU oracle for the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY: used by the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm, never by the product path.  It is
 * written straight from the method's definition, one step at a time, with no
 * blocking, fusion or reordering, so that it can be checked by eye:
 *
 *   1. p_i = softmax(l_i / T) for every one of the k+1 target rows
 *      ([DEE] §"O ciclo de rascunho e verificação"; [SD15] §"Why the result is
 *      exactly the target model", the accept_sampled signature).
 *   2. Judge the drafts left to right; accept x_i with probability
 *      min(1, p_i(x_i) / q_i(x_i)), i.e. accept iff p >= q or u < p/q
 *      ([DEE] §"A regra de amostragem por rejeição", rule 1; [SDF] §"El mecanismo
 *      desnudo", paso 3).  Stop at the first rejection.
 *   3. At a rejection draw from norm(max(0, p - q)); if all k survive draw a bonus
 *      token from p_k ([DEE] same section, rules 2 and 3; [SDF] paso 3).
 *   4. The categorical draw takes the first j whose running sum C_j exceeds
 *      u * C_{V-1} ([DEE] §"Amostragem especulativa em numpy, com prova": the
 *      sampler is a right-sided search of the cumulative sum).
 *   5. Greedy: accept while the draft equals argmax p, emit argmax at the first
 *      mismatch or for the bonus ([DEE] §"A regra de amostragem por rejeição",
 *      greedy paragraph; [SD15] §"Why the result is exactly the target model").
 *   6. num_accepted = n is the KV-cache length to keep ([DEE] §"O ciclo de
 *      rascunho e verificação", bookkeeping paragraph).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - an exact tie u == p/q rejects (strict "<", as in the page's sampler);
 *   - p >= q always accepts, which also covers q(x) == 0;
 *   - one uniform u_resample per sequence serves whichever single draw happens;
 *   - a rejected row whose residual has zero total mass draws from p instead;
 *   - a draw that runs past the last bin clamps to the last positive bin;
 *   - argmax ties go to the lowest index; positions after the draw are -1;
 *   - invalid data on a row or token the scan reaches marks the sequence invalid
 *     (num_accepted = -1, out all -1).
 *
 * Built with -ffp-contract=off so no multiply-add is fused and x86 / Arm builds
 * round identically.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Step 1: row statistics.  m = max_j l_j/T, S = sum_j exp(l_j/T - m), summed in
 * index order with Neumaier's compensation. */
int orc_row_stats(const double* l, double T, int V, double* m_out, double* S_out,
                  int32_t* argmax_out) {
    int bad = 0;
    int amax = -1;
    double lmax = -INFINITY;
    for (int j = 0; j < V; ++j) {
        double v = l[j];
        if (isnan(v) || v == INFINITY) bad = 1;
        if (v > lmax) { /* strict: the first (lowest) index of the maximum wins */
            lmax = v;
            amax = j;
        }
    }
    if (amax < 0) bad = 1; /* every entry -inf (or V == 0) */
    if (argmax_out) *argmax_out = amax < 0 ? 0 : amax;
    double m = lmax / T;
    double s = 0.0, c = 0.0;
    if (!bad) {
        for (int j = 0; j < V; ++j) {
            double e = exp(l[j] / T - m);
            double t = s + e;
            if (fabs(s) >= fabs(e)) c += (s - t) + e;
            else c += (e - t) + s;
            s = t;
        }
    }
    if (m_out) *m_out = m;
    if (S_out) *S_out = s + c;
    return bad;
}

/* p_j of a row from its statistics. */
static double row_p(const double* l, double T, double m, double S, int j) {
    return exp(l[j] / T - m) / S;
}

/* Weights of the draw at one row: the residual max(0, p - q) or p itself. */
static void draw_weights(const double* l, const double* q, double T, double m, double S,
                         int V, double* w) {
    for (int j = 0; j < V; ++j) {
        double p = row_p(l, T, m, S, j);
        if (q) w[j] = (p > q[j]) ? p - q[j] : 0.0;
        else w[j] = p;
    }
}

/* Step 4: first j with C_j > u * C_{V-1}, C_j the running sum in index order. */
static int categorical(const double* w, int V, double u, double* lo, double* hi,
                       int* overflow) {
    double C = 0.0;
    for (int j = 0; j < V; ++j) C += w[j];
    double Ctot = C;
    double tau = u * Ctot;
    double prev = 0.0;
    C = 0.0;
    for (int j = 0; j < V; ++j) {
        C += w[j];
        if (C > tau) {
            *lo = prev / Ctot;
            *hi = C / Ctot;
            *overflow = 0;
            return j;
        }
        prev = C;
    }
    /* Rounding pushed tau past the last boundary: clamp to the last positive bin. */
    *overflow = 1;
    int last = V - 1;
    while (last > 0 && !(w[last] > 0.0)) --last;
    C = 0.0;
    prev = 0.0;
    for (int j = 0; j <= last; ++j) {
        prev = C;
        C += w[j];
    }
    *lo = prev / Ctot;
    *hi = C / Ctot;
    return last;
}

int orc_draw_cdf(const double* l, const double* q, double T, int V, double* cdf) {
    double m, S;
    int32_t am;
    if (orc_row_stats(l, T, V, &m, &S, &am)) return 1;
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    draw_weights(l, q, T, m, S, V, w);
    double C = 0.0;
    for (int j = 0; j < V; ++j) C += w[j];
    double Ctot = C;
    if (!(Ctot > 0.0)) {
        free(w);
        return 1;
    }
    C = 0.0;
    for (int j = 0; j < V; ++j) {
        C += w[j];
        cdf[j] = C / Ctot;
    }
    free(w);
    return 0;
}

static void mark_invalid(int k, int32_t* out, int32_t* n_acc, int32_t* flags) {
    for (int i = 0; i <= k; ++i) out[i] = -1;
    *n_acc = -1;
    if (flags) *flags |= ORC_F_BAD;
}

/* Sample-and-match ([DEE] §"A regra de amostragem por rejeição", the simpler
 * exact scheme some engines use): at positions i = 0, 1, .. draw y_i from p_i
 * (the draw of step 4, with ua[i], or ur at position k) and keep the draft token
 * while y_i == x_i; the first position where they differ, or position k, emits
 * y_i.  Every emitted token is a draw from p, so the output is exact; a draft
 * survives position i with probability sum_v p_i(v) q_i(v).  A row, token or
 * uniform the scan reaches that is invalid invalidates the sequence.
 * *draw_lo / *draw_hi: the bin of the emitted draw. */
static void verify_match(const double* logits, const int32_t* x, const double* ua, double ur,
                         double T, int k, int V, int32_t* out, int32_t* n_acc,
                         double* draw_lo, double* draw_hi, int32_t* flags) {
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    int n = k, token = -1;
    for (int i = 0; i <= k; ++i) {
        const double* li = logits + (size_t)i * V;
        double m, S;
        int32_t am;
        if (orc_row_stats(li, T, V, &m, &S, &am)) {
            free(w);
            mark_invalid(k, out, n_acc, flags);
            return;
        }
        if (i < k && (x[i] < 0 || x[i] >= V)) {
            free(w);
            mark_invalid(k, out, n_acc, flags);
            return;
        }
        const double u = i < k ? ua[i] : ur;
        if (!(u >= 0.0 && u < 1.0)) {
            free(w);
            mark_invalid(k, out, n_acc, flags);
            return;
        }
        draw_weights(li, NULL, T, m, S, V, w);
        double lo, hi;
        int ovf;
        const int y = categorical(w, V, u, &lo, &hi, &ovf);
        if (ovf && flags) *flags |= ORC_F_OVERFLOW;
        if (i == k || y != x[i]) {
            n = i;
            token = y;
            if (draw_lo) *draw_lo = lo;
            if (draw_hi) *draw_hi = hi;
            break;
        }
    }
    free(w);
    for (int i = 0; i < n; ++i) out[i] = x[i];
    out[n] = token;
    for (int i = n + 1; i <= k; ++i) out[i] = -1;
    *n_acc = n;
}

/* Per-row statistics of one sequence supplied by the caller: the values step 1
 * (orc_row_stats) returned earlier for these same rows at the same T; rows i
 * of the sequence at index i. */
typedef struct {
    const double* m;
    const double* S;
    const int32_t* argmax;
    const int32_t* bad;
} given_stats;

/* Step 1 for row i: computed, or taken from `g` when the caller supplies it. */
static int stats_of(const double* li, double T, int V, const given_stats* g, int i, double* m,
                    double* S, int32_t* am) {
    if (!g) return orc_row_stats(li, T, V, m, S, am);
    *m = g->m[i];
    *S = g->S[i];
    *am = g->argmax[i];
    return g->bad[i];
}

static void verify_seq(int mode, const double* logits, const double* q, const int32_t* x,
                       const double* ua, double ur, double T, int k, int V, int32_t* out,
                       int32_t* n_acc, double* thr, double* draw_lo, double* draw_hi,
                       int32_t* flags, const given_stats* g);

void orc_verify_seq(int mode, const double* logits, const double* q, const int32_t* x,
                    const double* ua, double ur, double T, int k, int V,
                    int32_t* out, int32_t* n_acc, double* thr, double* draw_lo,
                    double* draw_hi, int32_t* flags) {
    verify_seq(mode, logits, q, x, ua, ur, T, k, V, out, n_acc, thr, draw_lo, draw_hi, flags,
               NULL);
}

static void verify_seq(int mode, const double* logits, const double* q, const int32_t* x,
                       const double* ua, double ur, double T, int k, int V, int32_t* out,
                       int32_t* n_acc, double* thr, double* draw_lo, double* draw_hi,
                       int32_t* flags, const given_stats* g) {
    if (mode == ORC_MATCH) {
        if (flags) *flags = 0;
        if (thr)
            for (int i = 0; i < k; ++i) thr[i] = NAN;
        if (draw_lo) *draw_lo = NAN;
        if (draw_hi) *draw_hi = NAN;
        verify_match(logits, x, ua, ur, T, k, V, out, n_acc, draw_lo, draw_hi, flags);
        return;
    }
    const int greedy = (mode == ORC_GREEDY);
    const double Tr = greedy ? 1.0 : T;
    if (flags) *flags = 0;
    if (thr)
        for (int i = 0; i < k; ++i) thr[i] = NAN;
    if (draw_lo) *draw_lo = NAN;
    if (draw_hi) *draw_hi = NAN;

    /* Step 2 (and 5): the left-to-right scan. */
    int n = k;
    for (int i = 0; i < k; ++i) {
        const double* li = logits + (size_t)i * V;
        double m, S;
        int32_t am;
        if (stats_of(li, Tr, V, g, i, &m, &S, &am)) {
            mark_invalid(k, out, n_acc, flags);
            return;
        }
        int xi = x[i];
        if (xi < 0 || xi >= V) {
            mark_invalid(k, out, n_acc, flags);
            return;
        }
        int accept;
        if (greedy) {
            accept = (xi == am);
        } else {
            double u = ua[i];
            double Q = q[(size_t)i * V + xi];
            if (!(u >= 0.0 && u < 1.0) || isnan(Q) || Q < 0.0) {
                mark_invalid(k, out, n_acc, flags);
                return;
            }
            double P = row_p(li, Tr, m, S, xi);
            if (thr) thr[i] = (P >= Q) ? 1.0 : P / Q;
            accept = (P >= Q) || (u < P / Q);
        }
        if (!accept) {
            n = i;
            break;
        }
    }

    /* Step 3 (and 5): the correction at the first rejection, or the bonus. */
    const double* ln = logits + (size_t)n * V;
    double m, S;
    int32_t am;
    if (stats_of(ln, Tr, V, g, n, &m, &S, &am)) {
        mark_invalid(k, out, n_acc, flags);
        return;
    }
    int token;
    if (greedy) {
        token = am;
    } else {
        if (!(ur >= 0.0 && ur < 1.0)) {
            mark_invalid(k, out, n_acc, flags);
            return;
        }
        double* w = (double*)malloc(sizeof(double) * (size_t)V);
        const double* qn = (n < k && mode == ORC_SAMPLE) ? q + (size_t)n * V : NULL;
        draw_weights(ln, qn, Tr, m, S, V, w);
        if (qn) {
            double tot = 0.0;
            for (int j = 0; j < V; ++j) tot += w[j];
            if (!(tot > 0.0)) { /* zero residual mass: draw from p */
                draw_weights(ln, NULL, Tr, m, S, V, w);
                if (flags) *flags |= ORC_F_DEGENERATE;
            }
        }
        double lo, hi;
        int ovf;
        token = categorical(w, V, ur, &lo, &hi, &ovf);
        if (ovf && flags) *flags |= ORC_F_OVERFLOW;
        if (draw_lo) *draw_lo = lo;
        if (draw_hi) *draw_hi = hi;
        free(w);
    }

    /* Step 6: outputs. */
    for (int i = 0; i < n; ++i) out[i] = x[i];
    out[n] = token;
    for (int i = n + 1; i <= k; ++i) out[i] = -1;
    *n_acc = n;
}

int orc_ngram_draft(const int32_t* history, const int32_t* lengths, int B, int Lmax, int k,
                    int n_min, int n_max, int32_t* draft, int32_t* num) {
    if (B < 0 || Lmax < 0 || k < 1 || n_min < 1 || n_max < n_min) return -1;
    if (B > 0 && (!history || !lengths || !draft || !num)) return -1;
    for (int b = 0; b < B; ++b) {
        const int32_t* h = history + (size_t)b * Lmax;
        int L = lengths[b];
        if (L < 0) L = 0;
        if (L > Lmax) L = Lmax;
        int best = -1;
        for (int n = n_max; n >= n_min && best < 0; --n) {
            if (L < n + 1) continue;
            for (int e = L - 2; e >= n - 1; --e) { /* most recent first */
                int t = 0;
                while (t < n && h[e - t] == h[L - 1 - t]) ++t;
                if (t == n) {
                    best = e;
                    break;
                }
            }
        }
        int32_t* d = draft + (size_t)b * k;
        int cnt = 0;
        if (best >= 0)
            for (int i = 0; i < k && best + 1 + i <= L - 1; ++i) d[cnt++] = h[best + 1 + i];
        for (int i = cnt; i < k; ++i) d[i] = -1;
        num[b] = cnt;
    }
    return 0;
}

static double bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int orc_verify_batch(int mode, const void* logits, int dtype, const float* q,
                     const int32_t* x, const float* ua, const float* ur, float T,
                     int B, int k, int V, int32_t* out, int32_t* n_acc,
                     double* row_m, double* row_S, int32_t* row_argmax,
                     double* row_px, double* row_qx, double* thr,
                     double* draw_lo, double* draw_hi, int32_t* flags, int nthreads) {
    if (B < 0 || k < 1 || V < 1 || !logits || !x || !out || !n_acc) return -1;
    if (dtype != 0 && dtype != 1) return -1;
    const int greedy = (mode == ORC_GREEDY);
    const int uses_q = (mode == ORC_SAMPLE || mode == ORC_SAMPLE_BUGGY);
    if (uses_q && !q) return -1;
    if (!greedy && (!ua || !ur)) return -1;
    const double Td = greedy ? 1.0 : (double)T;
    const size_t rowsz = (size_t)V;
    const size_t seqsz = (size_t)(k + 1) * rowsz;
    int nt = nthreads > 0 ? nthreads : orc_max_threads();
    (void)nt;

#pragma omp parallel num_threads(nt)
    {
        double* L = (double*)malloc(sizeof(double) * seqsz);
        double* Qd = uses_q ? (double*)malloc(sizeof(double) * (size_t)k * rowsz) : NULL;
        double* ua_d = (double*)malloc(sizeof(double) * (size_t)k);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            /* Step 0: exact conversion of the inputs to double. */
            if (dtype == 0) {
                const uint16_t* src = (const uint16_t*)logits + (size_t)b * seqsz;
                for (size_t j = 0; j < seqsz; ++j) L[j] = bf16_to_double(src[j]);
            } else {
                const float* src = (const float*)logits + (size_t)b * seqsz;
                for (size_t j = 0; j < seqsz; ++j) L[j] = (double)src[j];
            }
            if (uses_q) {
                const float* qs = q + (size_t)b * k * rowsz;
                for (size_t j = 0; j < (size_t)k * rowsz; ++j) Qd[j] = (double)qs[j];
            }
            if (!greedy)
                for (int i = 0; i < k; ++i) ua_d[i] = (double)ua[(size_t)b * k + i];
            /* Per-row statistics of every row, for parity of the stats. */
            for (int i = 0; i <= k; ++i) {
                size_t r = (size_t)b * (k + 1) + i;
                double m, S;
                int32_t am;
                int bad = orc_row_stats(L + (size_t)i * rowsz, Td, V, &m, &S, &am);
                if (row_m) row_m[r] = m;
                if (row_S) row_S[r] = bad ? NAN : S;
                if (row_argmax) row_argmax[r] = am;
                double px = NAN, qx = NAN;
                if (i < k) {
                    int xi = x[(size_t)b * k + i];
                    if (xi >= 0 && xi < V) {
                        if (!bad) px = row_p(L + (size_t)i * rowsz, Td, m, S, xi);
                        if (uses_q) qx = Qd[(size_t)i * rowsz + xi];
                    }
                }
                if (row_px) row_px[r] = px;
                if (row_qx) row_qx[r] = qx;
            }
            int32_t fl = 0;
            orc_verify_seq(mode, L, Qd, x + (size_t)b * k, ua_d, greedy ? 0.0 : (double)ur[b],
                           Td, k, V, out + (size_t)b * (k + 1), n_acc + b,
                           thr ? thr + (size_t)b * k : NULL, draw_lo ? draw_lo + b : NULL,
                           draw_hi ? draw_hi + b : NULL, &fl);
            if (flags) flags[b] = fl;
        }
        free(L);
        free(Qd);
        free(ua_d);
    }
    return 0;
}

/* Step 0 for one sequence: its k+1 logits rows and k q rows as doubles. */
static void seq_to_double(const void* logits, int dtype, const float* q, size_t b, size_t seqsz,
                          size_t qsz, double* L, double* Qd) {
    if (dtype == 0) {
        const uint16_t* src = (const uint16_t*)logits + b * seqsz;
        for (size_t j = 0; j < seqsz; ++j) L[j] = bf16_to_double(src[j]);
    } else {
        const float* src = (const float*)logits + b * seqsz;
        for (size_t j = 0; j < seqsz; ++j) L[j] = (double)src[j];
    }
    if (Qd) {
        const float* qs = q + b * qsz;
        for (size_t j = 0; j < qsz; ++j) Qd[j] = (double)qs[j];
    }
}

int orc_row_stats_batch(const void* logits, int dtype, float T, int R, int V, double* m,
                        double* S, int32_t* argmax, int32_t* bad, int nthreads) {
    if (R < 0 || V < 1 || !logits || !m || !S || !argmax || !bad) return -1;
    if (dtype != 0 && dtype != 1) return -1;
    int nt = nthreads > 0 ? nthreads : orc_max_threads();
    (void)nt;
#pragma omp parallel num_threads(nt)
    {
        double* L = (double*)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < R; ++r) {
            seq_to_double(logits, dtype, NULL, (size_t)r, (size_t)V, 0, L, NULL);
            bad[r] = orc_row_stats(L, (double)T, V, m + r, S + r, argmax + r);
        }
        free(L);
    }
    return 0;
}

int orc_verify_batch_stats(int mode, const void* logits, int dtype, const float* q,
                           const int32_t* x, const float* ua, const float* ur, float T, int B,
                           int k, int V, const double* st_m, const double* st_S,
                           const int32_t* st_argmax, const int32_t* st_bad, int32_t* out,
                           int32_t* n_acc, double* thr, double* draw_lo, double* draw_hi,
                           int32_t* flags, int nthreads) {
    if (B < 0 || k < 1 || V < 1 || !logits || !x || !out || !n_acc) return -1;
    if (!st_m || !st_S || !st_argmax || !st_bad) return -1;
    if (dtype != 0 && dtype != 1) return -1;
    if (mode != ORC_SAMPLE && mode != ORC_GREEDY && mode != ORC_SAMPLE_BUGGY) return -1;
    const int greedy = (mode == ORC_GREEDY);
    if (!greedy && (!q || !ua || !ur)) return -1;
    const double Td = greedy ? 1.0 : (double)T;
    const size_t seqsz = (size_t)(k + 1) * V, qsz = (size_t)k * V;
    int nt = nthreads > 0 ? nthreads : orc_max_threads();
    (void)nt;
#pragma omp parallel num_threads(nt)
    {
        double* L = (double*)malloc(sizeof(double) * seqsz);
        double* Qd = greedy ? NULL : (double*)malloc(sizeof(double) * qsz);
        double* ua_d = (double*)malloc(sizeof(double) * (size_t)k);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            seq_to_double(logits, dtype, q, (size_t)b, seqsz, qsz, L, Qd);
            if (!greedy)
                for (int i = 0; i < k; ++i) ua_d[i] = (double)ua[(size_t)b * k + i];
            const size_t r0 = (size_t)b * (k + 1);
            const given_stats g = {st_m + r0, st_S + r0, st_argmax + r0, st_bad + r0};
            int32_t fl = 0;
            verify_seq(mode, L, Qd, x + (size_t)b * k, ua_d, greedy ? 0.0 : (double)ur[b], Td, k,
                       V, out + (size_t)b * (k + 1), n_acc + b, thr ? thr + (size_t)b * k : NULL,
                       draw_lo ? draw_lo + b : NULL, draw_hi ? draw_hi + b : NULL, &fl, &g);
            if (flags) flags[b] = fl;
        }
        free(L);
        free(Qd);
        free(ua_d);
    }
    return 0;
}

/* ------------------------------------------------------------------ tree walk */

static void tree_invalid(int N, int32_t* out, int32_t* nodes, int32_t* n_acc,
                         int32_t* flags) {
    for (int i = 0; i < N; ++i) {
        out[i] = -1;
        nodes[i] = -1;
    }
    *n_acc = -1;
    if (flags) *flags |= ORC_F_BAD;
}

void orc_tree_seq(int mode, const double* logits, const double* q, const int32_t* tok,
                  const int32_t* par, const double* ua, double ur, double T, int N, int V,
                  int32_t* out, int32_t* nodes, int32_t* n_acc, double* thr, double* draw_lo,
                  double* draw_hi, int32_t* flags) {
    const int greedy = (mode == ORC_GREEDY);
    const double Tr = greedy ? 1.0 : T;
    if (flags) *flags = 0;
    if (thr)
        for (int j = 0; j < N; ++j) thr[j] = NAN;
    if (draw_lo) *draw_lo = NAN;
    if (draw_hi) *draw_hi = NAN;
    for (int j = 1; j < N; ++j)
        if (par[j] < 0 || par[j] >= j) {
            tree_invalid(N, out, nodes, n_acc, flags);
            return;
        }
    double* p = greedy ? NULL : (double*)malloc(sizeof(double) * (size_t)V);
    double* r = greedy ? NULL : (double*)malloc(sizeof(double) * (size_t)V);
    double* w = greedy ? NULL : (double*)malloc(sizeof(double) * (size_t)V);
    int cur = 0, n = 0, token = -1, bad = 0;
    for (;;) {
        const double* lc = logits + (size_t)cur * V;
        double m, S;
        int32_t am;
        if (orc_row_stats(lc, Tr, V, &m, &S, &am)) {
            bad = 1;
            break;
        }
        if (!greedy) {
            /* r = p, and w (the weights r is the normalisation of) = p too */
            for (int j = 0; j < V; ++j) {
                p[j] = row_p(lc, Tr, m, S, j);
                r[j] = p[j];
                w[j] = p[j];
            }
        }
        const double* qc = greedy ? NULL : q + (size_t)cur * V;
        int next = -1;
        for (int j = cur + 1; j < N && next < 0 && !bad; ++j) {
            if (par[j] != cur) continue;
            const int x = tok[j];
            if (x < 0 || x >= V) {
                bad = 1;
                break;
            }
            if (greedy) {
                if (x == am) next = j;
                continue;
            }
            const double u = ua[j], Q = qc[x], P = r[x];
            if (!(u >= 0.0 && u < 1.0) || isnan(Q) || Q < 0.0) {
                bad = 1;
                break;
            }
            if (thr) thr[j] = (P >= Q) ? 1.0 : P / Q;
            if (P >= Q || u < P / Q) {
                next = j;
                break;
            }
            /* rejected: r becomes the normalised residual max(0, r - q) */
            double Z = 0.0;
            for (int v = 0; v < V; ++v) {
                w[v] = (r[v] > qc[v]) ? r[v] - qc[v] : 0.0;
                Z += w[v];
            }
            if (mode == ORC_SAMPLE_BUGGY) {
                /* negative control: every sibling tested against p itself and
                   the residual taken once, as if each were a fresh chain step */
                for (int v = 0; v < V; ++v) w[v] = (p[v] > qc[v]) ? p[v] - qc[v] : 0.0;
                continue;
            }
            if (Z > 0.0) {
                for (int v = 0; v < V; ++v) r[v] = w[v] / Z;
            } else { /* zero residual mass: back to p */
                for (int v = 0; v < V; ++v) {
                    r[v] = p[v];
                    w[v] = p[v];
                }
                if (flags) *flags |= ORC_F_DEGENERATE;
            }
        }
        if (bad) break;
        if (next >= 0) {
            nodes[n] = next;
            out[n] = tok[next];
            ++n;
            cur = next;
            continue;
        }
        if (greedy) {
            token = am;
        } else {
            if (!(ur >= 0.0 && ur < 1.0)) {
                bad = 1;
                break;
            }
            double lo, hi;
            int ovf;
            token = categorical(w, V, ur, &lo, &hi, &ovf);
            if (ovf && flags) *flags |= ORC_F_OVERFLOW;
            if (draw_lo) *draw_lo = lo;
            if (draw_hi) *draw_hi = hi;
        }
        break;
    }
    free(p);
    free(r);
    free(w);
    if (bad) {
        tree_invalid(N, out, nodes, n_acc, flags);
        return;
    }
    out[n] = token;
    for (int i = n + 1; i < N; ++i) out[i] = -1;
    for (int i = n; i < N; ++i) nodes[i] = -1;
    *n_acc = n;
}

int orc_tree_batch(int mode, const void* logits, int dtype, const float* q, const int32_t* tok,
                   const int32_t* par, const float* ua, const float* ur, float T, int B, int N,
                   int V, int32_t* out, int32_t* nodes, int32_t* n_acc, double* row_m,
                   int32_t* row_argmax, double* thr, double* draw_lo, double* draw_hi,
                   int32_t* flags, int nthreads) {
    if (B < 0 || N < 1 || V < 1 || !logits || !tok || !par || !out || !nodes || !n_acc)
        return -1;
    if (dtype != 0 && dtype != 1) return -1;
    if (mode != ORC_SAMPLE && mode != ORC_GREEDY) return -1;
    const int greedy = (mode == ORC_GREEDY);
    if (!greedy && (!q || !ua || !ur)) return -1;
    const double Td = greedy ? 1.0 : (double)T;
    const size_t seqsz = (size_t)N * V;
    int nt = nthreads > 0 ? nthreads : orc_max_threads();
    (void)nt;
#pragma omp parallel num_threads(nt)
    {
        double* L = (double*)malloc(sizeof(double) * seqsz);
        double* Qd = greedy ? NULL : (double*)malloc(sizeof(double) * seqsz);
        double* ua_d = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            if (dtype == 0) {
                const uint16_t* src = (const uint16_t*)logits + (size_t)b * seqsz;
                for (size_t j = 0; j < seqsz; ++j) L[j] = bf16_to_double(src[j]);
            } else {
                const float* src = (const float*)logits + (size_t)b * seqsz;
                for (size_t j = 0; j < seqsz; ++j) L[j] = (double)src[j];
            }
            if (!greedy) {
                const float* qs = q + (size_t)b * seqsz;
                for (size_t j = 0; j < seqsz; ++j) Qd[j] = (double)qs[j];
                for (int j = 0; j < N; ++j) ua_d[j] = (double)ua[(size_t)b * N + j];
            }
            for (int i = 0; i < N; ++i) {
                double m, S;
                int32_t am;
                orc_row_stats(L + (size_t)i * V, Td, V, &m, &S, &am);
                if (row_m) row_m[(size_t)b * N + i] = m;
                if (row_argmax) row_argmax[(size_t)b * N + i] = am;
            }
            int32_t fl = 0;
            orc_tree_seq(mode, L, Qd, tok + (size_t)b * N, par + (size_t)b * N, ua_d,
                         greedy ? 0.0 : (double)ur[b], Td, N, V, out + (size_t)b * N,
                         nodes + (size_t)b * N, n_acc + b, thr ? thr + (size_t)b * N : NULL,
                         draw_lo ? draw_lo + b : NULL, draw_hi ? draw_hi + b : NULL, &fl);
            if (flags) flags[b] = fl;
        }
        free(L);
        free(Qd);
        free(ua_d);
    }
    return 0;
}
