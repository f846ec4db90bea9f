"""Pins of the float64 CPU oracle to what the pages and the mathematics fix.

Each test ties one part of the oracle to something other than itself: a value
printed on the pages (tests/golden, cited there), a closed form, a theorem
checked by exact enumeration, or a library routine in a special case.  A
plausible mistake anywhere in the oracle (a wrong residual, a swapped operand in
the acceptance ratio, a shifted draw index, a dropped temperature) fails at
least one of them; ``test_planted_mistakes_are_caught`` checks that directly.
"""
import math

import numpy as np
import pytest
from conftest import read_golden

from oracle import GREEDY, SAMPLE, SAMPLE_BUGGY, exact


def softmax64(l, T=1.0):
    z = np.asarray(l, dtype=np.float64) / T
    e = np.exp(z - z.max())
    return e / math.fsum(e)


# ---------------------------------------------------------------- row statistics

def test_row_stats_match_fsum(orc):
    """m and S against numpy max / exp and math.fsum (exactly rounded sum)."""
    g = np.random.default_rng(11)
    for V in (1, 2, 7, 33, 1000, 50000):
        for T in (0.5, 1.0, 1.7):
            l = g.normal(0, 3, V)
            m, S, am, bad = orc.row_stats(l, T)
            assert not bad
            z = l / T
            assert m == z.max()
            S_ref = math.fsum(np.exp(z - z.max()))
            assert abs(S - S_ref) <= 1e-14 * S_ref
            assert am == int(np.argmax(l))


def test_uniform_row_special_case(orc):
    """Equal logits: S = V exactly and every p_j = 1/V (draw = floor(u V))."""
    for V in (1, 3, 8, 1024):
        l = np.full(V, 0.375)
        m, S, am, bad = orc.row_stats(l, 0.9)
        assert S == V and am == 0 and not bad
        cdf = orc.draw_cdf(l, None, 0.9)
        assert np.allclose(cdf, np.arange(1, V + 1) / V, rtol=0, atol=1e-15)


def test_argmax_ties_lowest_index(orc):
    """Ties (common in bf16) go to the lowest index, as numpy.argmax does."""
    g = np.random.default_rng(5)
    for _ in range(200):
        V = int(g.integers(1, 40))
        l = g.integers(-3, 3, V).astype(np.float64)  # many ties
        assert orc.row_stats(l)[2] == int(np.argmax(l))


def test_invalid_rows(orc):
    for row in ([1.0, np.nan, 2.0], [1.0, np.inf], [-np.inf, -np.inf]):
        assert orc.row_stats(np.array(row))[3]
    assert not orc.row_stats(np.array([-np.inf, 0.0]))[3]


# ---------------------------------------------------------------- greedy

def test_greedy_equals_argmax_decoding(orc):
    """Greedy verify emits argmax p at every reached position and accepts exactly
    while the draft equals it ([DEE] greedy paragraph; [SD15] "identical to greedy")."""
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    for seed, dt in ((0, "bf16"), (1, "f32"), (2, "bf16")):
        inp = make_inputs(mode="greedy", B=64, k=5, V=300, dtype=dt, kind="zipf",
                          p_argmax=0.7, seed=seed)
        r = orc.verify_batch(GREEDY, inp.logits, dt, None, inp.x, None, None, 1.0)
        am = np.argmax(inp.logits_f32(), axis=2)
        for b in range(inp.B):
            n = r.n[b]
            match = inp.x[b] == am[b, :inp.k]
            n_ref = int(np.argmin(match)) if not match.all() else inp.k
            assert n == n_ref
            assert list(r.out[b, :n + 1]) == list(am[b, :n + 1])
            assert (r.out[b, n + 1:] == -1).all()


# ---------------------------------------------------------------- exact enumeration

def _random_case(g, k, V, T):
    logits = g.normal(0, 1.5, (k + 1, V))
    q = g.dirichlet(np.ones(V) * 0.7, size=k)
    return logits, q


@pytest.mark.parametrize("k,V", [(1, 2), (1, 5), (2, 3), (2, 4), (2, 5)])
def test_enumeration_reproduces_target(orc, k, V):
    """The emitted token at position i, jointly with reaching i, has probability
    prod_{j<i} alpha_j * p_i(b), exactly (the exactness argument of [DEE]
    §"A regra de amostragem por rejeição" and [SDF] §"Por qué la calidad no se degrada")."""
    g = np.random.default_rng(100 * k + V)
    for T in (1.0, 0.6):
        logits, q = _random_case(g, k, V, T)
        dist = exact.outcome_distribution(SAMPLE, logits, q, T)
        marg, en = exact.position_marginals(dist, k, V)
        p = np.array([softmax64(logits[i], T) for i in range(k + 1)])
        alpha = np.minimum(p[:k], q).sum(axis=1)
        reach = np.concatenate([[1.0], np.cumprod(alpha)])
        assert np.abs(marg - reach[:, None] * p).max() < 1e-12
        assert abs(en - reach[1:].sum()) < 1e-12
        assert abs(sum(float(v) for v in dist.values()) - 1.0) < 1e-12


def test_enumeration_catches_buggy_fallback(orc):
    """Negative control: resampling from p instead of the residual is biased
    ([DEE] "Júnior" aside; [SD15] §"Why the result is exactly the target model")."""
    g = np.random.default_rng(7)
    logits, q = _random_case(g, 2, 4, 1.0)
    dist = exact.outcome_distribution(SAMPLE_BUGGY, logits, q, 1.0)
    marg, _ = exact.position_marginals(dist, 2, 4)
    p = np.array([softmax64(r) for r in logits])
    alpha = np.minimum(p[:2], q).sum(axis=1)
    reach = np.concatenate([[1.0], np.cumprod(alpha)])
    assert np.abs(marg - reach[:, None] * p).max() > 1e-3


def test_greedy_enumeration(orc):
    """Greedy is the degenerate case: the output is argmax at every position."""
    g = np.random.default_rng(3)
    logits, q = _random_case(g, 2, 4, 1.0)
    dist = exact.outcome_distribution(GREEDY, logits, q, 1.0)
    am = logits.argmax(axis=1)
    for (out, n), pr in dist.items():
        assert list(out[:n + 1]) == list(am[:n + 1])
    reach1 = float(sum(pr for (out, n), pr in dist.items() if n >= 1))
    assert abs(reach1 - q[0, am[0]]) < 1e-12


@pytest.mark.parametrize("k,V", [(1, 3), (2, 4), (2, 5)])
def test_match_enumeration_reproduces_target(orc, k, V):
    """Sample-and-match ([DEE] §"A regra de amostragem por rejeição", the simpler
    exact scheme) is exact too: the emitted token at position i, jointly with
    reaching i, has probability prod_{j<i} beta_j * p_i(b), where a draft
    survives position j with probability beta_j = sum_v p_j(v) q_j(v), never
    more than rejection sampling's sum_v min(p_j(v), q_j(v))."""
    g = np.random.default_rng(300 + 10 * k + V)
    for T in (1.0, 0.7):
        logits, q = _random_case(g, k, V, T)
        dist = exact.match_outcome_distribution(logits, q, T)
        marg, en = exact.position_marginals(dist, k, V)
        p = np.array([softmax64(logits[i], T) for i in range(k + 1)])
        beta = (p[:k] * q).sum(axis=1)
        reach = np.concatenate([[1.0], np.cumprod(beta)])
        assert np.abs(marg - reach[:, None] * p).max() < 1e-12
        assert abs(en - reach[1:].sum()) < 1e-12
        assert abs(sum(float(v) for v in dist.values()) - 1.0) < 1e-12
        assert (beta <= np.minimum(p[:k], q).sum(axis=1) + 1e-15).all()


def test_match_toy_acceptance(orc):
    """On the page's seeded toy, sample-and-match keeps a draft with probability
    sum_v P[c, v] Q[c, v] = [0.245 0.270 0.321 0.316] per context c (the oracle's
    enumeration gives exactly that); the page's printed "0.39 to 0.55" does not
    reproduce from its own setup and is not used as a pin."""
    P, Q = exact.toy_bigram()
    beta = (P * Q).sum(axis=1)
    assert np.allclose(beta, [0.245, 0.270, 0.321, 0.316], atol=5e-4)
    for c in range(4):
        logits = np.log(np.stack([P[c], P[c]]))
        dist = exact.match_outcome_distribution(logits, Q[c][None, :], 1.0)
        accept = float(sum(pr for (out, n), pr in dist.items() if n >= 1))
        assert abs(accept - beta[c]) < 1e-12


# ---------------------------------------------------------------- the page's toy

def test_toy_alpha_matches_page(orc):
    """alpha per context printed on [DEE] §"Amostragem especulativa em numpy, com prova"."""
    want = [float(v) for v in read_golden("toy_alpha_per_context.txt")[0]]
    P, Q = exact.toy_bigram()
    got = []
    for c in range(4):
        rd = exact.toy_round_distribution(P, Q, c, k=1)
        got.append(float(sum(pr for new, pr in rd.items() if len(new) == 2)))
    assert [round(a, 3) for a in got] == want


def test_toy_tv_correct_and_buggy(orc):
    """Exact TV to the target joint: ~0 for the rejection rule, and the buggy rule's
    plateau the page reports (~0.107, sampled at N=1e5 and 4e5)."""
    P, Q = exact.toy_bigram()
    joint = exact.toy_exact_joint(P)
    rows = read_golden("toy_tv_table.txt")
    page_buggy = [float(tv) for n, s, tv in rows if s == "buggy" and int(n) >= 100000]
    for mode, lo, hi in ((SAMPLE, 0.0, 1e-12), (SAMPLE_BUGGY, None, None)):
        d = exact.toy_sequence_distribution(P, Q, k=3, L=4, mode=mode)
        tv = 0.5 * sum(abs(float(d.get(s, 0)) - p) for s, p in joint.items())
        if mode == SAMPLE:
            assert tv < hi
        else:
            # The sampled TV is the exact bias plus sampling noise of order 0.005 at
            # these N (the page's own target-only TV at N=4e5 is 0.0084).
            for v in page_buggy:
                assert abs(tv - v) < 0.005
            assert 0.100 < tv < 0.108


# ---------------------------------------------------------------- closed forms

def expected_tokens(alpha, k):
    """E[tokens per target pass] (Leviathan et al., quoted on [DEE] §"Quanto mais
    rápido: a matemática" and [SDF] §"La matemática que importa")."""
    return (1 - alpha ** (k + 1)) / (1 - alpha)


def test_closed_form_matches_page_tables():
    for k, a, _measured, formula in read_golden("tokens_per_call.txt"):
        # The page evaluates the formula at the unrounded measured alpha and prints
        # alpha to 3 decimals, so the printed value must lie inside the image of
        # [alpha - 0.0005, alpha + 0.0005] (E is increasing in alpha), +- rounding.
        lo = expected_tokens(float(a) - 0.0005, int(k)) - 0.0005
        hi = expected_tokens(float(a) + 0.0005, int(k)) + 0.0005
        assert lo <= float(formula) <= hi
    for a, gam, c, e_pr, s_pr in read_golden("worked_examples.txt"):
        e = expected_tokens(float(a), int(gam))
        assert abs(e - float(e_pr)) < 0.011  # the page rounds 3.288 -> 3.29, 4.152 -> 4.16
        assert round(e / (int(gam) * float(c) + 1), 2) == float(s_pr)
    ks = (1, 2, 3, 4, 5, 6, 8)
    for row in read_golden("speedup_table.txt"):
        c, a = float(row[0]), float(row[1])
        for kk, s in zip(ks, row[2:]):
            assert round(expected_tokens(a, kk) / (kk * c + 1), 2) == float(s)


@pytest.mark.parametrize("k", [1, 2])
def test_iid_mean_length_closed_form(orc, k):
    """With every position sharing p and q, E[n+1] = (1 - alpha^(k+1))/(1 - alpha)."""
    g = np.random.default_rng(21 + k)
    V = 4
    l = g.normal(0, 1, V)
    qrow = g.dirichlet(np.ones(V))
    logits = np.tile(l, (k + 1, 1))
    q = np.tile(qrow, (k, 1))
    dist = exact.outcome_distribution(SAMPLE, logits, q, 1.0)
    _, en = exact.position_marginals(dist, k, V)
    alpha = np.minimum(softmax64(l), qrow).sum()
    assert abs((en + 1) - expected_tokens(alpha, k)) < 1e-12


# ---------------------------------------------------------------- draw convention

def test_draw_matches_searchsorted_right(orc):
    """The categorical draw is the first j with C_j > u * C_{V-1} (a right-sided
    search of the running sum, [DEE] §"Amostragem especulativa em numpy, com prova"):
    checked against numpy.searchsorted on residual weights built with numpy, over a
    grid of u kept 1e-9 away from every boundary (the two sides' float64 roundings
    differ at ~1e-16); a dense sweep that includes the oracle's own boundaries never
    picks a zero-weight bin."""
    g = np.random.default_rng(9)
    checked = 0
    for trial in range(60):
        V = int(g.integers(2, 6))
        logits = g.normal(0, 1, (2, V))
        p0 = softmax64(logits[0])
        q0 = g.dirichlet(np.ones(V))
        if trial % 3 == 0:
            q0 = np.where(np.arange(V) % 2 == 0, p0 * 1.3, p0 * 0.2)
            q0 /= q0.sum()
        w = np.maximum(p0 - q0, 0.0)
        if w.sum() == 0:
            continue
        C = np.cumsum(w)
        # A draft that is rejected for sure: a token with p < q, u_accept just below 1.
        cand = [j for j in range(V) if p0[j] < q0[j]]
        if not cand:
            continue
        x = np.array([cand[0]], dtype=np.int32)
        nb = C[:-1] / C[-1]
        grid = [u for u in np.linspace(0, 1, 201)[:-1] if np.all(np.abs(nb - u) > 1e-9)]
        own = orc.draw_cdf(logits[0], q0, 1.0)
        for u in grid:
            r = orc.verify_seq(SAMPLE, logits, q0[None, :], x, np.array([1 - 1e-12]), u, 1.0)
            assert r.n == 0
            assert r.out[0] == int(np.searchsorted(C, u * C[-1], side="right"))
            checked += 1
        for u in [b for b in own if b < 1.0] + list(np.nextafter(own[own < 1.0], 0)):
            r = orc.verify_seq(SAMPLE, logits, q0[None, :], x, np.array([1 - 1e-12]), u, 1.0)
            assert w[r.out[0]] > 0
    assert checked > 1000


def test_draw_boundary_goes_right(orc):
    """With exactly representable weights (uniform logits, V a power of two, so
    p_j = 1/V exactly) a uniform landing on the boundary j/V draws token j: the
    right-sided convention of the page's sampler."""
    for V in (2, 4, 8):
        logits = np.zeros((2, V))
        q = np.full((1, V), 0.5 / V)  # p >= q: the draft is always accepted
        for j in range(V):
            r = orc.verify_seq(SAMPLE, logits, q, np.array([0]), np.array([0.5]), j / V, 1.0)
            assert r.n == 1 and r.out[1] == j
            assert r.draw_lo == j / V and r.draw_hi == (j + 1) / V


# ---------------------------------------------------------------- statistics

def _iid_batch(g, N, k, V, T, logits_row, qrow):
    logits = np.broadcast_to(logits_row.astype(np.float32), (N, k + 1, V)).copy()
    q = np.broadcast_to(qrow.astype(np.float32), (N, k, V)).copy()
    x = g.choice(V, size=(N, k), p=qrow.astype(np.float64) / qrow.astype(np.float64).sum())
    ua = g.random((N, k), dtype=np.float32)
    ur = g.random(N, dtype=np.float32)
    return logits, q, x.astype(np.int32), ua, ur


def _chi2_p(counts, probs):
    from scipy.stats import chi2
    n = counts.sum()
    exp_ = n * probs
    big = exp_ >= 5
    obs = list(counts[big]) + [counts[~big].sum()]
    ex = list(exp_[big]) + [exp_[~big].sum()]
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    stat = sum((o - e) ** 2 / e for o, e in zip(obs, ex))
    return chi2.sf(stat, len(ex) - 1)


def test_chi_square_million_trials(orc):
    """10^6 seeded verify calls on a config-1-shaped row (V=32, k=4, N(0, 2^2)
    logits, q from logits + N(0, 0.5^2)): every position's emitted token follows p
    (chi-square, cells with expected count < 5 pooled, as on [DEE] §"Amostragem
    especulativa em numpy, com prova"), the mean accepted length matches the closed
    form within 4 standard errors, and the buggy fallback fails at p < 1e-6."""
    g = np.random.default_rng(2024)
    V, k, T = 32, 4, 1.0
    l = (2.0 * g.standard_normal(V)).astype(np.float32)
    dl = l.astype(np.float64) + 0.5 * g.standard_normal(V)
    qrow = softmax64(dl).astype(np.float32)
    p = softmax64(l.astype(np.float64), T)
    alpha = float(np.minimum(p, qrow.astype(np.float64)).sum())
    N_total, chunk = 1_000_000, 100_000
    res = {}
    for mode in (SAMPLE, SAMPLE_BUGGY):
        counts = np.zeros((k + 1, V), dtype=np.int64)
        ns = []
        gg = np.random.default_rng(77)
        for _ in range(N_total // chunk):
            logits, q, x, ua, ur = _iid_batch(gg, chunk, k, V, T, l, qrow)
            r = orc.verify_batch(mode, logits, "f32", q, x, ua, ur, T)
            assert (r.n >= 0).all()
            ns.append(r.n.copy())
            for i in range(k + 1):
                col = r.out[:, i]
                counts[i] += np.bincount(col[col >= 0], minlength=V)
        res[mode] = (counts, np.concatenate(ns))
    counts, ns = res[SAMPLE]
    for i in range(k + 1):
        assert _chi2_p(counts[i], p) > 1e-4
    en = ns.mean()
    se = ns.std() / math.sqrt(ns.size)
    assert abs((en + 1) - expected_tokens(alpha, k)) < 4 * se
    counts_b, _ = res[SAMPLE_BUGGY]
    assert _chi2_p(counts_b[0], p) < 1e-6


# ---------------------------------------------------------------- edge cases

def test_edge_cases(orc):
    V, k = 5, 2
    l = np.log(np.array([[0.1, 0.2, 0.3, 0.15, 0.25]] * 3))
    q = np.array([[0.0, 0.5, 0.1, 0.2, 0.2]] * 2)
    # q(x) == 0 always accepts; p >= q always accepts
    r = orc.verify_seq(SAMPLE, l, q, np.array([0, 2]), np.array([0.999, 0.999]), 0.3, 1.0)
    assert r.n == 2 and list(r.out[:2]) == [0, 2] and r.thr[0] == 1.0
    # an exact tie u == p/q rejects
    pq = 0.2 / 0.5
    r = orc.verify_seq(SAMPLE, l, q, np.array([1, 2]), np.array([pq, 0.0]), 0.3, 1.0)
    assert r.n == 0
    # invalid token / uniform / row
    for x, ua, ur in (([5, 0], [0.1, 0.1], 0.3), ([0, 0], [1.0, 0.1], 0.3),
                      ([0, 0], [0.1, 0.1], 1.0)):
        r = orc.verify_seq(SAMPLE, l, q, np.array(x), np.array(ua), ur, 1.0)
        assert r.n == -1 and (r.out == -1).all() and r.flags & orc.F_BAD
    bad = l.copy()
    bad[0, 1] = np.nan
    r = orc.verify_seq(SAMPLE, bad, q, np.array([0, 0]), np.array([0.1, 0.1]), 0.3, 1.0)
    assert r.n == -1
    # a bad row after the first rejection is never read
    bad = l.copy()
    bad[2, 1] = np.nan
    r = orc.verify_seq(SAMPLE, bad, q, np.array([1, 0]), np.array([0.9, 0.1]), 0.3, 1.0)
    assert r.n == 0 and r.out[0] >= 0
    # zero residual mass at a rejection (q unnormalised, q >= p everywhere): draw from p
    q2 = np.array([[0.2, 0.4, 0.3, 0.15, 0.25]] * 2)
    r = orc.verify_seq(SAMPLE, l, q2, np.array([1, 0]), np.array([0.9, 0.1]), 0.05, 1.0)
    assert r.n == 0 and r.flags & orc.F_DEGENERATE and r.out[0] == 0
    # V == 1: always accept, bonus token 0
    r = orc.verify_seq(SAMPLE, np.zeros((3, 1)), np.ones((2, 1)), np.array([0, 0]),
                       np.array([0.5, 0.5]), 0.5, 1.0)
    assert r.n == 2 and list(r.out) == [0, 0, 0]


def test_planted_mistakes_are_caught(orc):
    """The buggy mode is a mistake planted in the oracle; the pins above must fail on
    it (they do: see test_enumeration_catches_buggy_fallback and the chi-square test).
    Here: a temperature the oracle ignored would fail the row-statistics pin."""
    l = np.array([0.3, 1.2, -0.7, 2.0])
    m1, S1, _, _ = orc.row_stats(l, 1.0)
    m2, S2, _, _ = orc.row_stats(l, 0.5)
    assert abs(S1 - S2) > 1e-3 and m2 == 2 * m1


# ---------------------------------------------------------------- n-gram drafter

def test_ngram_drafter_worked_cases(orc):
    """The prompt-lookup rule ([DEE] §"A família de rascunhos"; [SD15] §"What
    proposes the tokens"): the longest suffix n-gram (n_max down to n_min) that
    occurred before, its most recent occurrence, the tokens that followed it."""
    pad = -9
    cases = [
        # history, k, n_min, n_max, expected draft
        ([1, 2, 3, 4, 1, 2], 3, 1, 2, [3, 4, 1]),       # "1 2" seen at 0..1: copy 3 4 1
        ([1, 2, 3, 4, 1, 2], 5, 1, 2, [3, 4, 1, 2]),    # cut at the end of the history
        ([5, 6, 7, 8], 3, 1, 3, []),                    # nothing repeats: no draft
        ([7, 1, 9, 2, 9, 3, 9], 2, 1, 2, [3, 9]),       # "9" most recent earlier at 4 -> 3 9
        ([1, 2, 9, 5, 2, 9, 6, 2, 9], 2, 1, 2, [6, 2]),  # "2 9" at 4..5 (most recent) -> 6 2
        ([4, 2, 9, 5, 8, 2, 9], 3, 1, 3, [5, 8, 2]),    # "8 2 9" absent, "2 9" at 1..2
        ([3, 3, 3, 3], 2, 1, 2, [3]),                   # overlapping run: e = 2, one token left
        ([1], 2, 1, 1, []),                             # too short to hold an occurrence
    ]
    Lmax = max(len(c[0]) for c in cases)
    hist = np.full((len(cases), Lmax), pad, np.int32)
    for b, c in enumerate(cases):
        hist[b, :len(c[0])] = c[0]
    lens = np.array([len(c[0]) for c in cases], np.int32)
    for b, (h, k, n_min, n_max, want) in enumerate(cases):
        d, num = orc.ngram_draft(hist[b:b + 1], lens[b:b + 1], k, n_min, n_max)
        assert num[0] == len(want), (b, d, num)
        assert list(d[0, :num[0]]) == want and (d[0, num[0]:] == -1).all(), (b, d)


def test_ngram_drafter_periodic_stream(orc):
    """On a stream of period P >= n_max the draft is exactly the next k tokens of
    the period; on a stream without repeats it is empty."""
    g = np.random.default_rng(4)
    P, k = 11, 6
    period = g.permutation(1000)[:P].astype(np.int32)
    for L in (2 * P, 3 * P + 5, 5 * P - 1):
        h = np.resize(period, L)[None, :]
        d, num = orc.ngram_draft(h, np.array([L], np.int32), k, 1, 4)
        want = np.resize(period, L + k)[L:L + k]
        assert num[0] == k and np.array_equal(d[0], want)
    h = np.arange(50, dtype=np.int32)[None, :]
    d, num = orc.ngram_draft(h, np.array([50], np.int32), k, 1, 4)
    assert num[0] == 0 and (d == -1).all()


# ---------------------------------------------------------------- supplied statistics

@pytest.mark.parametrize("mode", [SAMPLE, GREEDY, SAMPLE_BUGGY])
def test_supplied_stats_batch_equals_plain_batch(orc, mode):
    """verify_batch_stats with the statistics of row_stats_batch gives, bit for
    bit, what verify_batch computes by itself: the supplied statistics are only
    step 1's own values, read instead of recomputed.  Invalid rows, tokens and
    uniforms are mixed in, and rows are scaled to T as the verify uses them."""
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    for dtype, V, T in (("f32", 37, 0.8), ("bf16", 1000, 1.3), ("f32", 5, 1.0)):
        inp = make_inputs(mode="greedy" if mode == GREEDY else "sample", B=64, k=5, V=V,
                          dtype=dtype, T=T, kind="zipf", draft_sigma=0.6, p_argmax=0.6,
                          seed=V)
        lg = inp.logits.copy()
        x = inp.x.copy()
        ua = None if inp.ua is None else inp.ua.copy()
        bad_val = 0x7FC0 if dtype == "bf16" else np.float32(np.nan)
        lg[3, 1, V // 2] = bad_val           # a NaN in a row the scan may reach
        lg[7, 0, :] = 0xFF80 if dtype == "bf16" else -np.inf  # an all -inf row
        x[9, 0] = V                           # a token out of range
        if ua is not None:
            ua[11, 0] = 1.0                   # a uniform out of range
        Tv = 1.0 if mode == GREEDY else T
        st = orc.row_stats_batch(lg, dtype, Tv)
        a = orc.verify_batch(mode, lg, dtype, inp.q, x, ua, inp.ur, Tv)
        b = orc.verify_batch_stats(mode, lg, dtype, inp.q, x, ua, inp.ur, Tv, st)
        assert np.array_equal(a.out, b.out) and np.array_equal(a.n, b.n)
        assert np.array_equal(a.flags, b.flags)
        for f in ("thr", "draw_lo", "draw_hi"):
            assert np.array_equal(getattr(a, f), getattr(b, f), equal_nan=True)
        # the supplied statistics are the batch's own per-row values
        assert np.array_equal(st.argmax, a.row_argmax)
        assert np.array_equal(st.m, a.row_m)
        assert np.array_equal(np.where(st.bad == 1, np.nan, st.S), a.row_S, equal_nan=True)
        assert (a.n < 0).sum() >= 2


def test_supplied_stats_are_read(orc):
    """The supplied statistics are really used: a planted change to one row's
    argmax changes the greedy outcome of that sequence and of no other."""
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    inp = make_inputs(mode="greedy", B=8, k=3, V=50, dtype="f32", kind="zipf", p_argmax=1.0,
                      seed=4)
    st = orc.row_stats_batch(inp.logits, "f32", 1.0)
    a = orc.verify_batch_stats(GREEDY, inp.logits, "f32", None, inp.x, None, None, 1.0, st)
    assert (a.n == 3).all()
    st.argmax[2, 1] = (st.argmax[2, 1] + 1) % 50
    b = orc.verify_batch_stats(GREEDY, inp.logits, "f32", None, inp.x, None, None, 1.0, st)
    assert b.n[2] == 1 and b.out[2, 1] == st.argmax[2, 1]
    assert np.array_equal(np.delete(a.out, 2, 0), np.delete(b.out, 2, 0))
