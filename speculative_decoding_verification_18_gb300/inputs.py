"""Seeded synthetic inputs for the verify step.

This module only makes inputs: target logits, the draft's distributions q, the
drafted tokens and the uniforms.  It holds none of the verify arithmetic (no
acceptance test, no residual, no categorical draw of the verifier); drafted
tokens are drawn with numpy's own ``Generator.choice``.  Both the CUDA path and
the CPU oracle are fed from here.

Workloads (sizes, value distributions and seeds):

  c1  sampled, B=1,   k=4, V=32,     fp32, T=1.0: target logits i.i.d. N(0, 2^2);
      draft logits = target + N(0, 0.5^2), q = softmax(draft logits).
  c2  greedy,  B=64,  k=4, V=32000,  bf16: Zipf-shaped rows (slope 1.1, N(0,1)
      noise) under a random vocabulary permutation; the draft token is the row's
      argmax with probability 0.8, else a uniform random id.
  c3  sampled, B=32,  k=5, V=128256, bf16, T=0.8: Zipf rows (1.1, N(0,1));
      q = softmax((logits + N(0, 0.7^2)) / 0.8).
  c4  sampled, B=256, k=8, V=151936, fp32, T=1.0: Zipf rows (1.0, N(0, 1.5^2));
      q = softmax(logits + N(0, 1)).
  c5  sampled, B=1,   k=8, V=256000, bf16, T=0.7: Zipf rows (1.1, N(0,1));
      q = softmax((logits + N(0, 0.5^2)) / 0.7).

A Zipf-shaped row puts -s*ln(r) + eps_r at the position pi(r-1) of a fresh random
permutation pi, r = 1..V.  Drafted tokens are sampled from the float32 q rows;
uniforms are float32 in [0, 1).  Every stream (logits, draft noise,
permutations, draft sampling, u_accept, u_resample) has its own child seed.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

WORKLOADS = {
    "c1": dict(mode="sample", B=1, k=4, V=32, dtype="f32", T=1.0, kind="gauss",
               scale=2.0, draft_sigma=0.5, draft_T=1.0, seed=0),
    "c2": dict(mode="greedy", B=64, k=4, V=32000, dtype="bf16", T=1.0, kind="zipf",
               slope=1.1, noise=1.0, p_argmax=0.8, seed=1),
    "c3": dict(mode="sample", B=32, k=5, V=128256, dtype="bf16", T=0.8, kind="zipf",
               slope=1.1, noise=1.0, draft_sigma=0.7, draft_T=0.8, seed=2),
    "c4": dict(mode="sample", B=256, k=8, V=151936, dtype="f32", T=1.0, kind="zipf",
               slope=1.0, noise=1.5, draft_sigma=1.0, draft_T=1.0, seed=3),
    "c5": dict(mode="sample", B=1, k=8, V=256000, dtype="bf16", T=0.7, kind="zipf",
               slope=1.1, noise=1.0, draft_sigma=0.5, draft_T=0.7, seed=4),
}

WORKLOAD_NAMES = {
    "c1": "sampled B=1 k=4 V=32 fp32 T=1.0 (gaussian logits)",
    "c2": "greedy B=64 k=4 V=32000 bf16 (zipf logits)",
    "c3": "sampled B=32 k=5 V=128256 bf16 T=0.8 (zipf logits)",
    "c4": "sampled B=256 k=8 V=151936 fp32 T=1.0 (zipf logits)",
    "c5": "sampled B=1 k=8 V=256000 bf16 T=0.7 (zipf logits)",
}


@dataclass
class VerifyInputs:
    mode: str                 # "sample" or "greedy"
    dtype: str                # "bf16" or "f32"
    B: int
    k: int
    V: int
    T: float
    logits: np.ndarray        # [B, k+1, V] uint16 bf16 bit patterns or float32
    q: np.ndarray | None      # [B, k, V] float32 (sampled) or None
    x: np.ndarray             # [B, k] int32 drafted tokens
    ua: np.ndarray | None     # [B, k] float32 u_accept
    ur: np.ndarray | None     # [B] float32 u_resample
    meta: dict = field(default_factory=dict)

    def logits_f32(self) -> np.ndarray:
        """The logits as float32 values (exact widening of bf16)."""
        if self.dtype == "bf16":
            return (self.logits.astype(np.uint32) << 16).view(np.float32)
        return self.logits

    @property
    def nbytes_logits(self) -> int:
        return int(self.logits.nbytes)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    names = ("logits", "draft_noise", "perm", "draft_sample", "u_accept", "u_resample")
    return dict(zip(names, ss.spawn(len(names))))


_CHUNK = 64


def _chunked(n_rows, seq: np.random.SeedSequence, fn):
    """Run fn(rng, r0, r1) over fixed 64-row chunks, each with its own child seed,
    on a thread pool (numpy releases the GIL); the result does not depend on the
    thread count."""
    starts = list(range(0, n_rows, _CHUNK))
    kids = seq.spawn(len(starts))
    workers = max(1, min(len(starts), os.cpu_count() or 1))

    def run(i):
        r0 = starts[i]
        fn(np.random.default_rng(kids[i]), r0, min(n_rows, r0 + _CHUNK))

    if workers == 1:
        for i in range(len(starts)):
            run(i)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(run, range(len(starts))))


def _zipf_rows(s_val, s_perm, n_rows, V, slope, noise):
    base = -slope * np.log(np.arange(1, V + 1, dtype=np.float64))
    out = np.empty((n_rows, V), dtype=np.float32)
    perm_kids = s_perm.spawn(-(-n_rows // _CHUNK))

    def fill(g, r0, r1):
        gp = np.random.default_rng(perm_kids[r0 // _CHUNK])
        vals = base[None, :] + noise * g.standard_normal((r1 - r0, V))
        perm = gp.permuted(np.tile(np.arange(V), (r1 - r0, 1)), axis=1)
        rows = np.empty((r1 - r0, V), dtype=np.float64)
        np.put_along_axis(rows, perm, vals, axis=1)
        out[r0:r1] = rows.astype(np.float32)

    _chunked(n_rows, s_val, fill)
    return out


def _draft_q(base_rows, s_noise, sigma, T):
    """q = softmax((target + N(0, sigma^2)) / T), rows in float64, stored float32."""
    n, V = base_rows.shape
    q = np.empty((n, V), dtype=np.float32)

    def fill(g, r0, r1):
        z = (base_rows[r0:r1].astype(np.float64) + sigma * g.standard_normal((r1 - r0, V))) / T
        z -= z.max(axis=1, keepdims=True)
        e = np.exp(z)
        q[r0:r1] = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)

    _chunked(n, s_noise, fill)
    return q


def make_inputs(mode="sample", B=1, k=4, V=32, dtype="f32", T=1.0, kind="zipf",
                slope=1.1, noise=1.0, scale=2.0, draft_sigma=0.5, draft_T=None,
                p_argmax=0.8, seed=0) -> VerifyInputs:
    """Build one seeded batch.  ``kind`` is "zipf" (Zipf-shaped rows) or "gauss"
    (i.i.d. N(0, scale^2) logits)."""
    if draft_T is None:
        draft_T = T
    s = _streams(seed)
    R = B * (k + 1)
    if kind == "zipf":
        rows = _zipf_rows(s["logits"], s["perm"], R, V, slope, noise)
    elif kind == "gauss":
        rows = (scale * np.random.default_rng(s["logits"]).standard_normal((R, V))).astype(
            np.float32)
    else:
        raise ValueError(kind)
    if dtype == "bf16":
        bits = bf16_bits(rows)
        logits = bits.reshape(B, k + 1, V)
        vals = (bits.astype(np.uint32) << 16).view(np.float32).reshape(B, k + 1, V)
    elif dtype == "f32":
        logits = rows.reshape(B, k + 1, V)
        vals = logits
    else:
        raise ValueError(dtype)

    if mode == "greedy":
        am = np.argmax(vals[:, :k, :], axis=2)
        gd = np.random.default_rng(s["draft_sample"])
        rnd = gd.integers(0, V, size=(B, k))
        keep = gd.random((B, k)) < p_argmax
        x = np.where(keep, am, rnd).astype(np.int32)
        return VerifyInputs(mode, dtype, B, k, V, float(T), logits, None, x, None, None,
                            meta=dict(kind=kind, seed=seed))

    q = _draft_q(vals[:, :k, :].reshape(B * k, V), s["draft_noise"], draft_sigma,
                 draft_T).reshape(B, k, V)
    x = np.empty((B, k), dtype=np.int32)
    gs = np.random.default_rng(s["draft_sample"])
    for b in range(B):
        for i in range(k):
            p = q[b, i].astype(np.float64)
            x[b, i] = gs.choice(V, p=p / p.sum())
    ua = np.random.default_rng(s["u_accept"]).random((B, k), dtype=np.float32)
    ur = np.random.default_rng(s["u_resample"]).random(B, dtype=np.float32)
    return VerifyInputs(mode, dtype, B, k, V, float(T), logits, q, x, ua, ur,
                        meta=dict(kind=kind, seed=seed))


def workload(name: str, seed: int | None = None) -> VerifyInputs:
    """One of the five named workloads (c1..c5), optionally with another seed."""
    cfg = dict(WORKLOADS[name])
    if seed is not None:
        cfg["seed"] = seed
    inp = make_inputs(**cfg)
    inp.meta["workload"] = name
    return inp


def toy_language(seed: int = 2, V: int = 4, keep: float = 0.55):
    """The bigram toy language of "Decodificação especulativa explicada", §"Amostragem
    especulativa em numpy, com prova": target rows P[t] = p(next | previous t) are
    Dirichlet(1) draws, and the draft blurs them, Q = keep * P + (1 - keep) * D with
    D another set of Dirichlet(1) rows.  The two draws are made with the page's
    generator calls in the page's order, the only order that reproduces its
    printed acceptance per context.  Returns float64 arrays P, Q of shape [V, V]."""
    g = np.random.default_rng(seed)
    P = g.dirichlet(np.ones(V), size=V)
    D = g.dirichlet(np.ones(V), size=V)
    return P, keep * P + (1.0 - keep) * D


def ngram_histories(B: int, Lmax: int, V: int = 32000, seed: int = 0, pool: int = 64,
                    p_phrase: float = 0.8, min_len: int | None = None):
    """Synthetic token streams that repeat themselves, for the n-gram drafter:
    each history concatenates pieces that are, with probability p_phrase, one of
    `pool` fixed phrases (3 to 12 tokens) and otherwise fresh random tokens (1 to
    8), to a length drawn uniformly in [min_len, Lmax] (default Lmax / 2).
    Returns (history [B, Lmax] int32 padded with -1, lengths [B] int32)."""
    g = np.random.default_rng(seed)
    phrases = [g.integers(0, V, size=int(g.integers(3, 13))).astype(np.int32) for _ in range(pool)]
    lo = Lmax // 2 if min_len is None else min_len
    hist = np.full((B, Lmax), -1, dtype=np.int32)
    lengths = g.integers(lo, Lmax + 1, size=B).astype(np.int32)
    for b in range(B):
        parts, n = [], 0
        while n < lengths[b]:
            if g.random() < p_phrase:
                piece = phrases[int(g.integers(0, pool))]
            else:
                piece = g.integers(0, V, size=int(g.integers(1, 9))).astype(np.int32)
            parts.append(piece)
            n += len(piece)
        row = np.concatenate(parts)[:lengths[b]] if parts else np.zeros(0, np.int32)
        hist[b, :len(row)] = row
    return hist, lengths


@dataclass
class TreeInputs:
    mode: str                 # "sample" or "greedy"
    dtype: str                # "bf16" or "f32"
    B: int
    N: int
    V: int
    T: float
    logits: np.ndarray        # [B, N, V] uint16 bf16 bit patterns or float32
    q: np.ndarray | None      # [B, N, V] float32: the draft distribution at each node
    tok: np.ndarray           # [B, N] int32 (entry 0 unused: -1)
    par: np.ndarray           # [B, N] int32 (entry 0: -1)
    ua: np.ndarray | None     # [B, N] float32
    ur: np.ndarray | None     # [B] float32
    meta: dict = field(default_factory=dict)


def tree_parents(N: int, branching=(4, 2, 2)) -> np.ndarray:
    """Parents of a tree built level by level (the shape of a Medusa-style static
    tree): the root has branching[0] children, each of those branching[1], and
    so on (the last entry repeats), nodes numbered breadth-first, cut at N."""
    par = [-1]
    level = [0]
    depth = 0
    while len(par) < N:
        nxt = []
        bf = branching[min(depth, len(branching) - 1)]
        for p in level:
            for _ in range(bf):
                if len(par) < N:
                    par.append(p)
                    nxt.append(len(par) - 1)
        if not nxt:
            break
        level = nxt
        depth += 1
    return np.asarray(par, dtype=np.int32)


def make_tree_inputs(mode="sample", B=1, N=16, V=32000, dtype="bf16", T=1.0,
                     branching=(4, 2, 2), random_shape=False, slope=1.1, noise=1.0,
                     draft_sigma=0.5, p_argmax=0.7, seed=0) -> TreeInputs:
    """A seeded batch of drafted trees.  Logits rows are Zipf-shaped as in
    make_inputs; the draft at node j is q_j = softmax((l_j + N(0, sigma^2)) / T);
    sampled: the children of node j are drawn independently from q_j; greedy:
    a node's first child is its argmax with probability p_argmax, the other
    children uniform tokens.  The shape is the level-by-level tree of
    ``branching`` for every sequence, or (random_shape) each node's parent
    uniform among the nodes before it."""
    s = _streams(seed)
    R = B * N
    rows = _zipf_rows(s["logits"], s["perm"], R, V, slope, noise)
    if dtype == "bf16":
        bits = bf16_bits(rows)
        logits = bits.reshape(B, N, V)
        vals = (bits.astype(np.uint32) << 16).view(np.float32).reshape(B, N, V)
    elif dtype == "f32":
        logits = rows.reshape(B, N, V)
        vals = logits
    else:
        raise ValueError(dtype)
    gt = np.random.default_rng(s["draft_sample"])
    if random_shape:
        par = np.full((B, N), -1, np.int32)
        for j in range(1, N):
            par[:, j] = gt.integers(0, j, B)
    else:
        par = np.tile(tree_parents(N, branching), (B, 1))
    tok = np.full((B, N), -1, np.int32)
    if mode == "greedy":
        am = np.argmax(vals, axis=2)
        for j in range(1, N):
            p = par[:, j]
            first = np.array([not (par[b, 1:j] == p[b]).any() for b in range(B)])
            keep = first & (gt.random(B) < p_argmax)
            tok[:, j] = np.where(keep, am[np.arange(B), p], gt.integers(0, V, B))
        return TreeInputs(mode, dtype, B, N, V, float(T), logits, None, tok, par, None, None,
                          meta=dict(seed=seed, branching=branching))
    q = _draft_q(vals.reshape(R, V), s["draft_noise"], draft_sigma, T).reshape(B, N, V)
    cdf = np.cumsum(q.astype(np.float64), axis=2)
    for j in range(1, N):
        c = cdf[np.arange(B), par[:, j]]
        u = gt.random(B) * c[:, -1]
        tok[:, j] = np.minimum((c <= u[:, None]).sum(axis=1), V - 1)
    ua = np.random.default_rng(s["u_accept"]).random((B, N), dtype=np.float32)
    ur = np.random.default_rng(s["u_resample"]).random(B, dtype=np.float32)
    return TreeInputs(mode, dtype, B, N, V, float(T), logits, q, tok, par, ua, ur,
                      meta=dict(seed=seed, branching=branching))


@dataclass
class Redraws:
    """Fresh drafts and uniforms for `reps` repetitions of one sampled batch."""
    x: np.ndarray    # [reps, B, k] int32, each x[r, b, i] drawn from q[b, i]
    ua: np.ndarray   # [reps, B, k] float32 in [0, 1)
    ur: np.ndarray   # [reps, B] float32 in [0, 1)


def redraw(inp: VerifyInputs, reps: int, seed: int) -> Redraws:
    """Seeded drafted tokens and uniforms for `reps` more verifies of the same
    logits and q: each repetition draws every x[b, i] afresh from the float32 row
    q[b, i] (numpy's ``Generator.choice``, as ``make_inputs`` does) and new
    u_accept / u_resample.  Many seeded rows then cost one logits tensor."""
    if inp.mode != "sample":
        raise ValueError("redraw needs a sampled batch")
    B, k, V = inp.B, inp.k, inp.V
    s = np.random.SeedSequence(seed).spawn(3)
    x = np.empty((reps, B, k), dtype=np.int32)
    qrows = inp.q.reshape(B * k, V)
    kids = s[0].spawn(B * k)

    def fill(g, r0, r1):
        for r in range(r0, r1):
            p = qrows[r].astype(np.float64)
            gr = np.random.default_rng(kids[r])
            x[:, r // k, r % k] = gr.choice(V, size=reps, p=p / p.sum())

    _chunked(B * k, s[1].spawn(1)[0], fill)
    ua = np.random.default_rng(s[1]).random((reps, B, k), dtype=np.float32)
    ur = np.random.default_rng(s[2]).random((reps, B), dtype=np.float32)
    return Redraws(x, ua, ur)
