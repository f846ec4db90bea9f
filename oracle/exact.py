"""Exact enumeration over the oracle: the pins that need no sampling.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The verify step is a deterministic function of its inputs once the uniforms are
fixed, and piecewise constant in those uniforms: an accept decision flips only at
u_accept = min(1, p/q), and the draw changes bin only at a boundary C_j / C_{V-1}.
So cutting u-space into cells at every such boundary and calling the oracle once
at each cell's midpoint gives the exact probability of every outcome, weighted by
the cell volumes and by the draft-token probabilities prod_i q_i(x_i).

Theorem being pinned ([DEE] §"A regra de amostragem por rejeição", the exactness
argument; [SDF] §"Por qué la calidad no se degrada"): the token emitted at every
position i, given that positions 0..i-1 were accepted, is distributed exactly as
p_i, and position i is reached with probability prod_{j<i} alpha_j,
alpha_j = sum_x min(p_j(x), q_j(x)).
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

from . import GREEDY, MATCH, SAMPLE, draw_cdf, verify_seq


def _cells(bounds):
    """Cells [a, b) of [0, 1) cut at the sorted unique interior points of ``bounds``."""
    pts = sorted({0.0, 1.0, *[float(b) for b in bounds if 0.0 < b < 1.0]})
    return [(a, b) for a, b in zip(pts[:-1], pts[1:]) if b > a]


def outcome_distribution(mode, logits, q, T=1.0):
    """Exact distribution of (out tokens, n) for one sequence whose drafts x_i ~ q_i.

    logits: [k+1, V] float64; q: [k, V] float64 (rows summing to 1).  Returns a dict
    {(tuple(out), n): Fraction probability}.
    """
    logits = np.asarray(logits, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k1, V = logits.shape
    k = k1 - 1
    # Boundaries of the draw at every possible decision row: residual and plain p
    # (the union refines both, so the same cells serve the negative control too).
    draw_bounds = []
    for i in range(k + 1):
        b = []
        for qq in ((q[i] if i < k else None), None):
            c = draw_cdf(logits[i], qq, T)
            if c is not None:
                b.extend(c.tolist())
        draw_bounds.append(_cells(b))
    dist = {}
    for x in itertools.product(range(V), repeat=k):
        wx = Fraction(1)
        for i, xi in enumerate(x):
            wx *= Fraction(float(q[i, xi]))
        if wx == 0:
            continue
        # Accept thresholds of every position: with all u_accept = 0 each position
        # with p > 0 accepts, so the oracle reports min(1, P/Q) for all of them.
        probe = verify_seq(mode, logits, q, x, np.zeros(k), 0.5, T)
        thr = probe.thr
        # Cells of u_accept: per position, [0, a) accepts and [a, 1) rejects.
        per_pos = []
        for i in range(k):
            a = 0.0 if mode == GREEDY else float(thr[i])
            cells = [c for c in _cells([a]) if c[1] > c[0]]
            if mode == GREEDY:
                cells = [(0.0, 1.0)]
            per_pos.append(cells)
        for ucells in itertools.product(*per_pos):
            wu = Fraction(1)
            ua = np.empty(k)
            for i, (a, b) in enumerate(ucells):
                wu *= Fraction(b) - Fraction(a)
                ua[i] = 0.5 * (a + b)
            # Which row decides depends only on ua; probe it, then cut u_resample.
            first = verify_seq(mode, logits, q, x, ua, 0.5, T)
            if first.n < 0:
                raise RuntimeError("oracle marked a valid enumeration input invalid")
            rcells = [(0.0, 1.0)] if mode == GREEDY else draw_bounds[first.n]
            for (a, b) in rcells:
                res = verify_seq(mode, logits, q, x, ua, 0.5 * (a + b), T)
                key = (tuple(int(t) for t in res.out), res.n)
                dist[key] = dist.get(key, Fraction(0)) + wx * wu * (Fraction(b) - Fraction(a))
    return dist


def match_outcome_distribution(logits, q, T=1.0):
    """Exact distribution of (out tokens, n) under sample-and-match for one
    sequence whose drafts x_i ~ q_i ([DEE] §"A regra de amostragem por
    rejeição", the simpler exact scheme).  The uniform of each position's draw
    ranges over the cells of that row's bins, so every outcome is enumerated with
    its exact probability.  Same layout and result type as outcome_distribution.
    """
    logits = np.asarray(logits, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k1, V = logits.shape
    k = k1 - 1
    cells = [_cells(draw_cdf(logits[i], None, T).tolist()) for i in range(k + 1)]
    dist = {}
    for x in itertools.product(range(V), repeat=k):
        wx = Fraction(1)
        for i, xi in enumerate(x):
            wx *= Fraction(float(q[i, xi]))
        if wx == 0:
            continue
        for ucells in itertools.product(*cells):
            wu = Fraction(1)
            u = np.empty(k + 1)
            for i, (a, b) in enumerate(ucells):
                wu *= Fraction(b) - Fraction(a)
                u[i] = 0.5 * (a + b)
            res = verify_seq(MATCH, logits, None, x, u[:k], u[k], T)
            if res.n < 0:
                raise RuntimeError("oracle marked a valid enumeration input invalid")
            key = (tuple(int(t) for t in res.out), res.n)
            dist[key] = dist.get(key, Fraction(0)) + wx * wu
    return dist


def position_marginals(dist, k, V):
    """P(out_i = b and position i reached) as a float64 array [k+1, V], and E[n]."""
    marg = [[Fraction(0)] * V for _ in range(k + 1)]
    en = Fraction(0)
    for (out, n), pr in dist.items():
        en += n * pr
        for i, t in enumerate(out):
            if t >= 0:
                marg[i][t] += pr
    return np.array([[float(v) for v in row] for row in marg]), float(en)


def toy_bigram(seed: int = 2, V: int = 4, keep: float = 0.55):
    """The V=4 bigram toy language of [DEE] §"Amostragem especulativa em numpy, com prova".

    Target rows P[t] are Dirichlet(1) draws; the draft blurs them as
    Q = keep * P + (1 - keep) * (independent Dirichlet(1) rows).  The generator
    calls come in the page's order so the printed alpha per context reproduces.
    """
    g = np.random.default_rng(seed)
    P = g.dirichlet(np.ones(V), size=V)
    noise = g.dirichlet(np.ones(V), size=V)
    Q = keep * P + (1.0 - keep) * noise
    return P, Q


def toy_round_distribution(P, Q, prev, k, mode=SAMPLE):
    """Exact distribution of the tokens one speculative round appends after ``prev``.

    The draft proposes x_1..x_k autoregressively from Q (x_i ~ Q[x_{i-1}], x_0 =
    prev); the target scores rows P[prev], P[x_1], .., P[x_k] in one pass
    ([DEE] §"O ciclo de rascunho e verificação").  Target rows enter the oracle
    as logits ln P with T = 1.
    """
    V = P.shape[0]
    lnP = np.log(P)
    out = {}
    for x in itertools.product(range(V), repeat=k):
        ctx = [prev] + list(x[:-1])
        wx = Fraction(1)
        for c, t in zip(ctx, x):
            wx *= Fraction(float(Q[c, t]))
        logits = lnP[[prev] + list(x)]
        qrows = Q[ctx]
        # Condition on the drafts: enumerate only the uniforms.
        sub = _outcomes_given_drafts(mode, logits, qrows, x)
        for new, pr in sub.items():
            out[new] = out.get(new, Fraction(0)) + wx * pr
    return out


def _outcomes_given_drafts(mode, logits, q, x):
    k = len(x)
    probe = verify_seq(mode, logits, q, x, np.zeros(k), 0.5, 1.0)
    per_pos = [_cells([float(probe.thr[i])]) for i in range(k)]
    res_map = {}
    for ucells in itertools.product(*per_pos):
        wu = Fraction(1)
        ua = np.empty(k)
        for i, (a, b) in enumerate(ucells):
            wu *= Fraction(b) - Fraction(a)
            ua[i] = 0.5 * (a + b)
        first = verify_seq(mode, logits, q, x, ua, 0.5, 1.0)
        n = first.n
        b = []
        for qq in ((q[n] if n < k else None), None):
            c = draw_cdf(logits[n], qq, 1.0)
            if c is not None:
                b.extend(c.tolist())
        for (a, bb) in _cells(b):
            res = verify_seq(mode, logits, q, x, ua, 0.5 * (a + bb), 1.0)
            new = tuple(int(t) for t in res.out[: res.n + 1])
            res_map[new] = res_map.get(new, Fraction(0)) + wu * (Fraction(bb) - Fraction(a))
    return res_map


def toy_sequence_distribution(P, Q, k=3, L=4, bos=0, mode=SAMPLE):
    """Exact distribution over the V**L length-L sequences of the multi-round loop
    of [DEE] §"Amostragem especulativa em numpy, com prova" (rounds are appended
    and the result is truncated to L tokens)."""
    V = P.shape[0]
    rounds = {p: toy_round_distribution(P, Q, p, k, mode) for p in range(V)}
    done = {}
    frontier = {(): Fraction(1)}
    while frontier:
        nxt = {}
        for seq, pr in frontier.items():
            prev = seq[-1] if seq else bos
            for new, pn in rounds[prev].items():
                s = seq + new
                if len(s) >= L:
                    s = s[:L]
                    done[s] = done.get(s, Fraction(0)) + pr * pn
                else:
                    nxt[s] = nxt.get(s, Fraction(0)) + pr * pn
        frontier = nxt
    return done


def toy_exact_joint(P, L=4, bos=0):
    """Plain target-only probabilities of every length-L sequence."""
    V = P.shape[0]
    joint = {}
    for seq in itertools.product(range(V), repeat=L):
        pr, prev = 1.0, bos
        for t in seq:
            pr *= P[prev, t]
            prev = t
        joint[seq] = pr
    return joint
