"""Pins of the oracle's tree walk (CPU).

Tree verification checks several drafted continuations at once ("Decodificação
especulativa explicada", §"A família de rascunhos", Medusa's tree attention;
"Speculative decoding: el secretario...", §"Tree attention").  The pages give
no rule; the oracle takes the plainest exact one (greedy: follow the child that
equals the argmax; sampled: recursive rejection over each node's children,
which were drawn independently from the node's draft distribution).  Pinned by:
- reduction to the chain rule (pinned elsewhere) when every node has one child;
- the greedy walk's defining properties, checked with numpy's argmax;
- exactness of the sampled walk by exact enumeration: the emitted token at the
  root is distributed as p_root, and the token after an accepted child c as p_c
  (the property the pages demand of any speculative scheme: the target's
  distribution is unchanged);
- invalid inputs.
"""
import itertools

import numpy as np
import pytest

import oracle


def _chain_tree(k):
    par = np.r_[-1, np.arange(k)].astype(np.int32)
    return par


@pytest.mark.parametrize("seed", range(40))
def test_chain_reduction_sampled(seed):
    g = np.random.default_rng(seed)
    k, V = int(g.integers(1, 6)), int(g.integers(2, 9))
    T = float(g.uniform(0.5, 1.5))
    l = g.normal(0, 2, (k + 1, V))
    q = g.dirichlet(np.ones(V), size=k)
    if seed % 3 == 0:
        q[:, 0] = 0.0
        q /= q.sum(axis=1, keepdims=True)
    x = g.integers(0, V, k).astype(np.int32)
    ua = g.random(k)
    ur = float(g.random())
    a = oracle.verify_seq(oracle.SAMPLE, l, q, x, ua, ur, T)
    tok = np.r_[-1, x].astype(np.int32)
    qt = np.vstack([q, np.full((1, V), 0.5)])
    b = oracle.tree_seq(oracle.SAMPLE, l, qt, tok, _chain_tree(k), np.r_[0.0, ua], ur, T)
    assert b.n == a.n
    assert np.array_equal(b.out[:k + 1], a.out)
    assert np.array_equal(b.nodes[:a.n], np.arange(1, a.n + 1))
    judged = ~np.isnan(a.thr)
    assert np.array_equal(b.thr[1:][judged], a.thr[judged])
    assert (b.draw_lo, b.draw_hi) == (a.draw_lo, a.draw_hi)


@pytest.mark.parametrize("seed", range(20))
def test_chain_reduction_greedy(seed):
    g = np.random.default_rng(100 + seed)
    k, V = int(g.integers(1, 6)), int(g.integers(2, 9))
    l = np.round(g.normal(0, 1, (k + 1, V)), 1)  # ties
    am = l.argmax(axis=1)
    x = np.where(g.random(k) < 0.7, am[:k], g.integers(0, V, k)).astype(np.int32)
    a = oracle.verify_seq(oracle.GREEDY, l, None, x, None, None, 1.0)
    b = oracle.tree_seq(oracle.GREEDY, l, None, np.r_[-1, x], _chain_tree(k), None, None, 1.0)
    assert b.n == a.n and np.array_equal(b.out[:k + 1], a.out)


def _random_tree(g, N):
    par = np.full(N, -1, np.int32)
    for j in range(1, N):
        par[j] = int(g.integers(0, j))
    return par


@pytest.mark.parametrize("seed", range(30))
def test_greedy_walk_properties(seed):
    """Each accepted node is a child of the previous one (the root first) whose
    token is that node's argmax, and no earlier sibling carries it; the walk
    stops at a node none of whose children carries its argmax; the emitted token
    is that argmax."""
    g = np.random.default_rng(200 + seed)
    N, V = int(g.integers(1, 12)), int(g.integers(2, 6))
    l = np.round(g.normal(0, 1, (N, V)), 1)
    par = _random_tree(g, N)
    am = l.argmax(axis=1)
    tok = np.full(N, -1, np.int32)
    for j in range(1, N):  # drafts that often equal the parent's argmax
        tok[j] = am[par[j]] if g.random() < 0.5 else int(g.integers(0, V))
    r = oracle.tree_seq(oracle.GREEDY, l, None, tok, par, None, None, 1.0)
    cur = 0
    for i in range(r.n):
        c = int(r.nodes[i])
        assert par[c] == cur and tok[c] == am[cur] and r.out[i] == tok[c]
        sib = [j for j in range(1, c) if par[j] == cur]
        assert all(tok[j] != am[cur] for j in sib)
        cur = c
    assert all(tok[j] != am[cur] for j in range(1, N) if par[j] == cur)
    assert r.out[r.n] == am[cur]
    assert (r.out[r.n + 1:] == -1).all() and (r.nodes[r.n:] == -1).all()


def _softmax(l, T):
    z = np.exp(l / T - np.max(l / T))
    return z / z.sum()


@pytest.mark.parametrize("seed", range(4))
def test_sampled_walk_is_exact(seed):
    """Root with two children drawn independently from q_0, node 1 with two
    children drawn from q_1, node 2 a leaf (V = 3).  Over every draft outcome
    (weights q_0(x1) q_0(x2) q_1(x3) q_1(x4)) and every uniform cell: the first
    emitted token follows p_0 and, given node 1 accepted, the next follows p_1."""
    g = np.random.default_rng(300 + seed)
    V, N, T = 3, 5, float(g.uniform(0.6, 1.4))
    l = g.normal(0, 1.5, (N, V))
    q = g.dirichlet(np.ones(V), size=N)
    par = np.array([-1, 0, 0, 1, 1], np.int32)
    p0, p1 = _softmax(l[0], T), _softmax(l[1], T)
    first = np.zeros(V)
    second = np.zeros(V)
    reach1 = 0.0
    total = 0.0
    for x1, x2, x3, x4 in itertools.product(range(V), repeat=4):
        wx = q[0, x1] * q[0, x2] * q[1, x3] * q[1, x4]
        tok = np.array([-1, x1, x2, x3, x4], np.int32)
        for (nodes, outs), w in _enumerate_nodes(l, q, tok, par, T).items():
            total += wx * w
            first[outs[0]] += wx * w
            if nodes[0] == 1:
                reach1 += wx * w
                second[outs[1]] += wx * w
    assert abs(total - 1.0) < 1e-12
    np.testing.assert_allclose(first, p0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(second / reach1, p1, rtol=0, atol=1e-12)


def _enumerate_nodes(l, q, tok, par, T, mode=None):
    """Exact outcome distribution of the sampled walk for fixed drafts, keyed by
    (accepted nodes, emitted tokens).  The walk is piecewise constant in the
    uniforms, so u-space is cut at the thresholds the oracle reports (a tested
    child j accepts iff ua[j] < thr[j]) and at the bin edges of the final draw
    ([draw_lo, draw_hi) is the bin of the drawn token), recursively, and the
    oracle is evaluated at cell midpoints."""
    N = len(tok)
    dist = {}

    mode = oracle.SAMPLE if mode is None else mode

    def run(ua, ur):
        return oracle.tree_seq(mode, l, q, tok, par, ua, ur, T)

    def rec(fixed, weight):
        ua = np.full(N, 0.5)
        for j, v in fixed.items():
            ua[j] = v
        r = run(ua, 0.5)
        free = [j for j in range(1, N) if not np.isnan(r.thr[j]) and j not in fixed]
        if free:
            j = free[0]
            t = float(r.thr[j])
            for a, b in ((0.0, t), (t, 1.0)):
                if b > a:
                    rec({**fixed, j: 0.5 * (a + b)}, weight * (b - a))
            return
        todo = [(0.0, 1.0)]
        while todo:
            a, b = todo.pop()
            rr = run(ua, 0.5 * (a + b))
            lo, hi = max(a, rr.draw_lo), min(b, rr.draw_hi)
            key = (tuple(int(v) for v in rr.nodes), tuple(int(v) for v in rr.out))
            dist[key] = dist.get(key, 0.0) + weight * (hi - lo)
            if lo > a:
                todo.append((a, lo))
            if b > hi:
                todo.append((hi, b))

    rec({}, 1.0)
    return dist


def test_enumeration_catches_a_plausible_mistake():
    """Negative control: testing every sibling against p itself (no residual
    update between siblings) breaks exactness, and the enumeration sees it."""
    g = np.random.default_rng(7)
    V, N, T = 3, 3, 1.0
    l = g.normal(0, 1.5, (N, V))
    q = g.dirichlet(np.ones(V), size=N)
    par = np.array([-1, 0, 0], np.int32)
    p0 = _softmax(l[0], T)
    for mode, exact in ((oracle.SAMPLE, True), (oracle.SAMPLE_BUGGY, False)):
        first = np.zeros(V)
        for x1, x2 in itertools.product(range(V), repeat=2):
            wx = q[0, x1] * q[0, x2]
            tok = np.array([-1, x1, x2], np.int32)
            for (nodes, outs), w in _enumerate_nodes(l, q, tok, par, T, mode).items():
                first[outs[0]] += wx * w
        err = np.abs(first - p0).max()
        assert (err < 1e-12) == exact, (mode, err)


def test_invalid_inputs():
    g = np.random.default_rng(9)
    N, V = 5, 4
    l = g.normal(size=(N, V))
    q = g.dirichlet(np.ones(V), size=N)
    par = np.array([-1, 0, 0, 1, 1], np.int32)
    tok = np.array([-1, 1, 2, 0, 3], np.int32)
    ua = np.full(N, 0.99)
    ok = oracle.tree_seq(oracle.SAMPLE, l, q, tok, par, ua, 0.3, 1.0)
    assert ok.n >= 0
    bad_par = par.copy()
    bad_par[3] = 3
    r = oracle.tree_seq(oracle.SAMPLE, l, q, tok, bad_par, ua, 0.3, 1.0)
    assert r.n == -1 and (r.out == -1).all() and r.flags & oracle.F_BAD
    bad_tok = tok.copy()
    bad_tok[1] = V
    r = oracle.tree_seq(oracle.SAMPLE, l, q, bad_tok, par, ua, 0.3, 1.0)
    assert r.n == -1
    bad_u = ua.copy()
    bad_u[1] = 1.0
    assert oracle.tree_seq(oracle.SAMPLE, l, q, tok, par, bad_u, 0.3, 1.0).n == -1
    assert oracle.tree_seq(oracle.SAMPLE, l, q, tok, par, ua, 1.5, 1.0).n == -1
    bad_q = q.copy()
    bad_q[0, 1] = np.nan
    assert oracle.tree_seq(oracle.SAMPLE, l, bad_q, tok, par, ua, 0.3, 1.0).n == -1
    # a bad row the walk never reaches is not read: node 2 after node 1 accepts
    l2 = l.copy()
    l2[2, 0] = np.nan
    ua0 = np.zeros(N)  # node 1 accepted at the root, node 3 at node 1
    r = oracle.tree_seq(oracle.SAMPLE, l2, q, tok, par, ua0, 0.3, 1.0)
    assert r.n == 2 and list(r.nodes[:2]) == [1, 3]
    # a single-node tree: only the draw at the root
    r = oracle.tree_seq(oracle.SAMPLE, l[:1], q[:1], tok[:1], par[:1], ua[:1], 0.3, 1.0)
    assert r.n == 0 and r.out[0] >= 0
