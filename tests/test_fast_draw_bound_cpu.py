"""The fast draw's certificate against adversarial exponentials (CPU).

The GPU's fast draw ("Decodificação especulativa explicada", §"A regra de
amostragem por rejeição": the residual norm(max(0, p - q)) at a rejection, p
itself for the bonus; the categorical rule of §"Amostragem especulativa em
numpy, com prova") forms each p from one fp32 hardware exponential whose
relative error is only bounded (1.75e-7, checked exhaustively on the GPU)
and whose exponent is otherwise exact to first order (l - m by TwoSum, the
product's rounding and log2(e)/T's low part recovered),
sums the positive elements' y and q without rounding error that matters, and
keeps its token only when u C lies farther from each edge of the chosen bin
than that edge's error bound (the errors before the edge weighed by 1 - u,
those after it by u).  This test restates that arithmetic in Python: float32
values by rounding float64 ones, the sums exactly (integers at a fine scale),
the normaliser with an adversarial error of the size its pairwise chunk sums
allow, and the exponential as the exact 2^a times (1 + s E) with the sign s of
each element chosen adversarially (against a particular bin edge, or at
random).  It checks that a certified token is always the token of the exact
draw (the oracle's, in float64, far more accurate than any margin D), that most
draws away from edges are certified, and that the same emulation with D cut to
a quarter does certify wrong tokens (so the test can see a bound that is too
small).
"""
import math

import numpy as np
import pytest

E = 1.75e-7                    # the assumed worst relative error of ex2.approx (kEx2RelErr)
U = 2.0 ** -24
K_EY = E + 1.0625 * U          # kFastEy
K_HI, K_LO = 1 + 2.0 ** -12, 1 - 2.0 ** -12
K_UND = 3.9e-4
LN2F = float(np.float32(0.693147181))
SCALE = 200                    # exact integer sums at 2^-200


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _ints(v):
    """Exact integers v 2^SCALE of float values (all finite, >= 2^-150 or 0)."""
    return [int(math.ldexp(x, SCALE)) for x in v]


def _sum8(v):
    """sum8: ((v0+v1)+(v2+v3)) + ((v4+v5)+(v6+v7)) in float32."""
    f = np.float32
    return float(f(f(f(v[0] + v[1]) + f(v[2] + v[3])) + f(f(v[4] + v[5]) + f(v[6] + v[7]))))


def _prefix8(v, e):
    """prefix8: the pairwise prefix of 8 float32 values up to element e."""
    f = np.float32
    n01, n45 = f(v[0] + v[1]), f(v[4] + v[5])
    n03 = f(n01 + f(v[2] + v[3]))
    if e < 4:
        return float([f(v[0]), n01, f(n01 + v[2]), n03][e])
    part = [f(v[4]), n45, f(n45 + v[6]), f(n45 + f(v[6] + v[7]))][e - 4]
    return float(f(n03 + part))


def emulate_fast_draw(l, q, T, u, s_row, signs, d_scale=1.0, s_sign=1.0, exact=True):
    """The fast draw's arithmetic on one row.  l: logits (float32 values), q:
    the draft row or None (bonus draw), s_row: the row stream's normaliser,
    signs: +1 / -1 per element for the exponential's error, s_sign: the sign of
    the normaliser's own rounding; exact: the float-float chunk sums (summed
    exactly here), else the pairwise float32 ones.  Returns (token, certified)
    or None when the pass would hand the draw to the precise pass."""
    V = l.size
    m = float(l.max())
    v = 1.4426950408889634 / T
    chi = float(np.float32(v))
    clo = float(np.float32(v - chi))
    d = l - m                           # exact in float64 (float32 operands)
    dh = f32(d)                         # TwoSum: the float32 difference and its error
    dl = d - dh
    a = f32(dh * chi)
    # the exponent's residual (the product's rounding, c's low part, the
    # difference's error), applied to first order; its own roundings are far
    # below 2^-33 of y
    t = ((dh * chi - a) + dh * clo + dl * chi) * math.log(2.0)
    with np.errstate(over="ignore", invalid="ignore"):
        y0 = np.where(a >= -126.0, f32(np.exp2(a) * (1.0 + signs * E)), 0.0)
    y = np.where(y0 > 0, f32(y0 * t + y0), 0.0)
    if q is None:
        pos = np.ones(V, bool)
        und = np.zeros(V, bool)
        qv = np.zeros(V)
    else:
        qv = q.astype(np.float64)
        ih = float(np.float32(1.0 / float(np.float32(float(np.float32(s_row)) * K_HI))))
        il = float(np.float32(1.0 / float(np.float32(float(np.float32(s_row)) * K_LO))))
        pos = f32(y * ih) > qv
        zero = f32(y * il) < qv
        und = ~pos & ~zero
    yp = np.where(pos, y, 0.0)
    qp = np.where(pos, qv, 0.0)
    rest = float(y[~pos].sum())
    if exact:
        # C in units of 2^-62 of p from exact sums (the float-float chunk sums
        # are exact to ~2^-44, far below the bound)
        Yi = np.cumsum(np.array(_ints(yp), dtype=object))
        Qi = np.cumsum(np.array(_ints(qp), dtype=object))
        S_int = int(Yi[-1]) + int(math.ldexp(rest * (1 + s_sign * 3 * U), SCALE))
        Cy = [int(x) for x in Yi]
        Cq = [int(x) >> (SCALE - 62) for x in Qi]
        num = lambda Y: (Y << 62)
    else:
        # chunk sums pairwise in float32, then fixed point (Y: 2^-EY, Q: 2^-62)
        S_row32 = float(np.float32(s_row))
        ey = max(0, min(61, 61 - math.frexp(S_row32)[1]))
        pad = (-V) % 8
        ypp = np.concatenate([yp, np.zeros(pad)]).astype(np.float32)
        qpp = np.concatenate([qp, np.zeros(pad)]).astype(np.float32)
        Cy, Cq, by, bq = [], [], 0, 0
        for c in range(0, V, 8):
            for e in range(min(8, V - c)):
                Cy.append(by + int(math.ldexp(_prefix8(ypp[c:c + 8], e), ey)))
                Cq.append(bq + int(math.ldexp(_prefix8(qpp[c:c + 8], e), 62)))
            by += int(math.ldexp(_sum8(ypp[c:c + 8]), ey))
            bq += int(math.ldexp(_sum8(qpp[c:c + 8]), 62))
        Yall = by
        S_int = (Yall << (SCALE - ey)) + int(math.ldexp(rest * (1 + s_sign * 3 * U), SCALE))
        num = lambda Y: (Y << (62 + SCALE - ey))
    Sd = math.ldexp(S_int, -SCALE)
    if not (Sd > 0 and abs(Sd - s_row) <= Sd / 8192):
        return None
    C = [num(Y) // S_int - Qc for Y, Qc in zip(Cy, Cq)]
    Ctot = C[-1]
    if Ctot <= 0:
        return None
    tau = (int(math.ldexp(float(np.float32(u)), 40)) * Ctot) >> 40  # u has 24 bits: exact
    tok = next(j for j in range(V) if yp[j] > 0 and C[j] > tau)
    lo = C[tok - 1] if tok > 0 else 0
    hi = C[tok]
    # the certificate: each edge's own bound, the errors before the edge
    # weighed by 1 - u and those after it by u
    Ptot = num(Cy[-1]) // S_int
    Qtot = Cq[-1]
    Ppos = Ptot * 2.0 ** -62
    eS = K_EY + 3 * U * (max(0.0, 1.0 - Ppos) if exact else 1.0)
    kP = (K_EY + (0.0 if exact else 3 * U)) * 1.004
    kQ = (0.0 if exact else 3 * U) * 1.004
    Dc = K_UND * qv[und].sum() * 1.004 * 2.0 ** 62 + 2.0 ** 20 + 2.0 * (V / 8) + 64.0
    uQ = (int(math.ldexp(float(np.float32(u)), 40)) * Qtot) >> 40
    if exact:
        cm = 0.0
    else:
        c0 = (tok // 8) * 8
        cm = float(num(int(math.ldexp(_sum8(ypp[c0:c0 + 8]), ey))) // S_int
                   + int(math.ldexp(_sum8(qpp[c0:c0 + 8]), 62)))

    def edge(Yb, Qb):
        Pb = num(Yb) // S_int
        dp = (kP * ((1 - u) * Pb + u * max(Ptot - Pb, 0))
              + kQ * ((1 - u) * Qb + u * max(Qtot - Qb, 0) + 2 * cm)
              + eS * 1.004 * (abs(uQ - Qb) + 1 + (hi - lo))
              + max(u, 1.0 - u) * Dc + 2.0) * d_scale
        return int(min(dp, 4.0e18)) + 1

    Dlo = edge(Cy[tok - 1], Cq[tok - 1]) if tok > 0 else edge(0, 0)
    Dhi = edge(Cy[tok], Cq[tok])
    return tok, (tau - lo >= Dlo and hi - tau > Dhi)


def exact_cdf(orc, l, q, T):
    return orc.draw_cdf(l.astype(np.float64), None if q is None else q.astype(np.float64), T)


def _rows(seed, n):
    """Zipf-shaped rows (the workloads' shape) with a draft q from noisy logits."""
    g = np.random.default_rng(seed)
    for _ in range(n):
        V = int(g.integers(300, 3000))
        T = float(g.choice([0.7, 0.8, 1.0, 1.3]))
        base = -1.05 * np.log(np.arange(1, V + 1)) + g.normal(0, 1.2, V)
        l = f32(g.permutation(base))
        z = (l + g.normal(0, 0.7, V)) / T
        qq = np.exp(z - z.max())
        q = (qq / qq.sum()).astype(np.float32)
        yield g, l, q, T


def _sweep(orc, d_scale, seed, n_rows=12, exact=True):
    """Draws at uniforms placed around bin edges, with the exponential's errors
    signed against each edge; returns (certified, certified and wrong, total)."""
    cert = wrong = total = 0
    for g, l, q, T in _rows(seed, n_rows):
        for qrow in (q, None):
            cdf = exact_cdf(orc, l, qrow, T)
            if cdf is None:
                continue
            z = l.astype(np.float64) / T
            S = float(np.exp(z - z.max()).sum())
            # edges where the bins on both sides carry weight
            w = np.diff(np.concatenate([[0.0], cdf]))
            cand = np.flatnonzero((w > 1e-6) & (np.roll(w, -1) > 1e-6))
            cand = cand[(cand > 0) & (cand < l.size - 1)]
            if cand.size == 0:
                continue
            for edge in g.choice(cand, size=min(4, cand.size), replace=False):
                for pattern in ("before+", "before-", "random"):
                    if pattern == "random":
                        signs = g.choice([-1.0, 1.0], l.size)
                    else:
                        sgn = 1.0 if pattern == "before+" else -1.0
                        signs = np.where(np.arange(l.size) <= edge, sgn, -sgn)
                    s_row = S * (1 + float(g.uniform(-2.0 ** -14, 2.0 ** -14)))
                    s_sign = float(g.choice([-1.0, 1.0]))
                    c = float(cdf[edge])
                    for off in np.geomspace(2e-9, 3e-6, 9):
                        for u in (c - off, c + off):
                            u = float(np.float32(u))
                            if not 0.0 <= u < 1.0:
                                continue
                            r = emulate_fast_draw(l, qrow, T, u, s_row, signs, d_scale, s_sign,
                                                  exact)
                            if r is None:
                                continue
                            total += 1
                            tok, ok = r
                            exact = int(np.searchsorted(cdf, u, side="right"))
                            if ok:
                                cert += 1
                                wrong += tok != exact
    return cert, wrong, total


@pytest.mark.parametrize("exact", [True, False], ids=["float-float", "pairwise"])
def test_certified_tokens_are_exact(orc, exact):
    cert, wrong, total = _sweep(orc, 1.0, seed=12, exact=exact)
    assert total > 1000
    assert wrong == 0, f"{wrong} certified tokens differ from the exact draw"
    assert cert > 0.15 * total  # the certificate is not vacuous near edges


def test_certificate_far_from_edges(orc):
    """Uniforms drawn at random: almost every draw is certified, and correctly."""
    n = ok = 0
    for g, l, q, T in _rows(5, 12):
        cdf = exact_cdf(orc, l, q, T)
        z = l.astype(np.float64) / T
        S = float(np.exp(z - z.max()).sum())
        for _ in range(20):
            u = float(np.float32(g.random()))
            r = emulate_fast_draw(l, q, T, u, S, g.choice([-1.0, 1.0], l.size))
            if r is None:
                continue
            n += 1
            tok, c = r
            if c:
                ok += 1
                assert tok == int(np.searchsorted(cdf, u, side="right"))
    assert n > 200 and ok > 0.9 * n


@pytest.mark.parametrize("exact", [True, False], ids=["float-float", "pairwise"])
def test_a_quarter_of_the_bound_certifies_wrong_tokens(orc, exact):
    """Planted mistake: the same emulation with D cut to a quarter certifies
    wrong tokens on the adversarial sweep, so the sweep above can see a bound
    that is too small."""
    _, wrong, _ = _sweep(orc, 0.25, seed=12, exact=exact)
    assert wrong > 0
