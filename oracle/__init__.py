"""Plain float64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package; the product
path (the CUDA library and its binding) never does, and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, float64, OpenMP over sequences);
this module only builds it with gcc and marshals numpy arrays through ctypes.
``enumerate_exact`` (in ``exact.py``) adds the exact-enumeration checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

SAMPLE, GREEDY, SAMPLE_BUGGY, MATCH = 0, 1, 2, 3
F_BAD, F_DEGENERATE, F_OVERFLOW = 1, 2, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, -O2, OpenMP, no FMA contraction)."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                             os.path.getmtime(os.path.join(HERE, "oracle.h")))):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(LIB)
    P = ctypes.c_void_p
    lib.orc_row_stats.argtypes = [P, ctypes.c_double, ctypes.c_int, P, P, P]
    lib.orc_row_stats.restype = ctypes.c_int
    lib.orc_draw_cdf.argtypes = [P, P, ctypes.c_double, ctypes.c_int, P]
    lib.orc_draw_cdf.restype = ctypes.c_int
    lib.orc_verify_seq.argtypes = [ctypes.c_int, P, P, P, P, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_int, ctypes.c_int, P, P, P, P, P, P]
    lib.orc_verify_seq.restype = None
    lib.orc_verify_batch.argtypes = [ctypes.c_int, P, ctypes.c_int, P, P, P, P, ctypes.c_float,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                     P, P, P, P, P, P, P, P, P, ctypes.c_int]
    lib.orc_verify_batch.restype = ctypes.c_int
    lib.orc_ngram_draft.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, P, P]
    lib.orc_ngram_draft.restype = ctypes.c_int
    lib.orc_row_stats_batch.argtypes = [P, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                        ctypes.c_int, P, P, P, P, ctypes.c_int]
    lib.orc_row_stats_batch.restype = ctypes.c_int
    lib.orc_verify_batch_stats.argtypes = [ctypes.c_int, P, ctypes.c_int, P, P, P, P,
                                           ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, P, P, P, P, P, P, P, P, P, P,
                                           ctypes.c_int]
    lib.orc_verify_batch_stats.restype = ctypes.c_int
    lib.orc_max_threads.argtypes = []
    lib.orc_max_threads.restype = ctypes.c_int
    lib.orc_tree_seq.argtypes = [ctypes.c_int, P, P, P, P, P, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P]
    lib.orc_tree_seq.restype = None
    lib.orc_tree_batch.argtypes = [ctypes.c_int, P, ctypes.c_int, P, P, P, P, P, ctypes.c_float,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P,
                                   P, P, P, ctypes.c_int]
    lib.orc_tree_batch.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().orc_max_threads())


def row_stats(l, T: float = 1.0):
    """(m, S, argmax, bad) of one float64 row."""
    l = np.ascontiguousarray(l, dtype=np.float64)
    m = np.zeros(1)
    S = np.zeros(1)
    am = np.zeros(1, dtype=np.int32)
    bad = _load().orc_row_stats(_ptr(l), float(T), l.size, _ptr(m), _ptr(S), _ptr(am))
    return float(m[0]), float(S[0]), int(am[0]), bool(bad)


def draw_cdf(l, q=None, T: float = 1.0):
    """Normalised cumulative boundaries C_j / C_{V-1} of the draw weights of one row."""
    l = np.ascontiguousarray(l, dtype=np.float64)
    qq = None if q is None else np.ascontiguousarray(q, dtype=np.float64)
    cdf = np.zeros(l.size)
    rc = _load().orc_draw_cdf(_ptr(l), _ptr(qq), float(T), l.size, _ptr(cdf))
    return None if rc else cdf


@dataclass
class SeqResult:
    out: np.ndarray
    n: int
    thr: np.ndarray
    draw_lo: float
    draw_hi: float
    flags: int


def verify_seq(mode, logits, q, x, ua, ur, T) -> SeqResult:
    """One sequence with float64 inputs: logits [k+1,V], q [k,V], x [k], ua [k], ur."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    k1, V = logits.shape
    k = k1 - 1
    x = np.ascontiguousarray(x, dtype=np.int32)
    qq = None if q is None else np.ascontiguousarray(q, dtype=np.float64)
    uu = None if ua is None else np.ascontiguousarray(ua, dtype=np.float64)
    out = np.zeros(k + 1, dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    thr = np.zeros(k)
    lo = np.zeros(1)
    hi = np.zeros(1)
    fl = np.zeros(1, dtype=np.int32)
    _load().orc_verify_seq(int(mode), _ptr(logits), _ptr(qq), _ptr(x), _ptr(uu),
                           float(0.0 if ur is None else ur), float(T), k, V, _ptr(out),
                           _ptr(n), _ptr(thr), _ptr(lo), _ptr(hi), _ptr(fl))
    return SeqResult(out, int(n[0]), thr, float(lo[0]), float(hi[0]), int(fl[0]))


@dataclass
class BatchResult:
    out: np.ndarray        # [B, k+1] int32
    n: np.ndarray          # [B] int32
    row_m: np.ndarray      # [B, k+1] max_j l_j / T
    row_S: np.ndarray      # [B, k+1] sum_j exp(l_j/T - m)
    row_argmax: np.ndarray  # [B, k+1]
    row_px: np.ndarray     # [B, k+1] p_i(x_i) (NaN on row k)
    row_qx: np.ndarray     # [B, k+1] q_i(x_i) (NaN on row k)
    thr: np.ndarray        # [B, k] min(1, P/Q) at judged positions, NaN elsewhere
    draw_lo: np.ndarray    # [B]
    draw_hi: np.ndarray    # [B]
    flags: np.ndarray      # [B]


def verify_batch(mode, logits, dtype: str, q, x, ua, ur, T, nthreads: int = 0) -> BatchResult:
    """Batch verify over inputs in the device layouts.

    logits: [B, k+1, V] uint16 bf16 bit patterns (dtype "bf16") or float32 ("f32");
    q: [B, k, V] float32 or None (greedy, sample-and-match); x: [B, k] int32;
    ua: [B, k] float32; ur: [B] float32 (sample-and-match: the draws at positions
    0..k-1 and k).
    """
    B, k1, V = logits.shape
    k = k1 - 1
    if dtype == "bf16":
        logits = np.ascontiguousarray(logits, dtype=np.uint16)
        dt = 0
    elif dtype == "f32":
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        dt = 1
    else:
        raise ValueError(dtype)
    greedy = mode == GREEDY
    qq = np.ascontiguousarray(q, dtype=np.float32) if mode in (SAMPLE, SAMPLE_BUGGY) else None
    x = np.ascontiguousarray(x, dtype=np.int32)
    uu = None if greedy else np.ascontiguousarray(ua, dtype=np.float32)
    rr = None if greedy else np.ascontiguousarray(ur, dtype=np.float32)
    r = BatchResult(
        out=np.zeros((B, k + 1), np.int32), n=np.zeros(B, np.int32),
        row_m=np.zeros((B, k + 1)), row_S=np.zeros((B, k + 1)),
        row_argmax=np.zeros((B, k + 1), np.int32), row_px=np.zeros((B, k + 1)),
        row_qx=np.zeros((B, k + 1)), thr=np.zeros((B, k)), draw_lo=np.zeros(B),
        draw_hi=np.zeros(B), flags=np.zeros(B, np.int32))
    rc = _load().orc_verify_batch(
        int(mode), _ptr(logits), dt, _ptr(qq), _ptr(x), _ptr(uu), _ptr(rr), float(T), B, k, V,
        _ptr(r.out), _ptr(r.n), _ptr(r.row_m), _ptr(r.row_S), _ptr(r.row_argmax),
        _ptr(r.row_px), _ptr(r.row_qx), _ptr(r.thr), _ptr(r.draw_lo), _ptr(r.draw_hi),
        _ptr(r.flags), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r


def _logits_arg(logits, dtype: str):
    if dtype == "bf16":
        return np.ascontiguousarray(logits, dtype=np.uint16), 0
    if dtype == "f32":
        return np.ascontiguousarray(logits, dtype=np.float32), 1
    raise ValueError(dtype)


@dataclass
class RowStats:
    m: np.ndarray       # [B, k+1] max_j l_j / T
    S: np.ndarray       # [B, k+1] sum_j exp(l_j/T - m)
    argmax: np.ndarray  # [B, k+1]
    bad: np.ndarray     # [B, k+1] 1 for an invalid row


def row_stats_batch(logits, dtype: str, T: float, nthreads: int = 0) -> RowStats:
    """Step 1 on every row of logits [B, k+1, V] (device layout) at temperature T."""
    B, k1, V = logits.shape
    lg, dt = _logits_arg(logits, dtype)
    st = RowStats(np.zeros((B, k1)), np.zeros((B, k1)), np.zeros((B, k1), np.int32),
                  np.zeros((B, k1), np.int32))
    rc = _load().orc_row_stats_batch(_ptr(lg), dt, float(T), B * k1, V, _ptr(st.m), _ptr(st.S),
                                     _ptr(st.argmax), _ptr(st.bad), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return st


def verify_batch_stats(mode, logits, dtype: str, q, x, ua, ur, T, stats: RowStats,
                       nthreads: int = 0) -> BatchResult:
    """verify_batch (modes SAMPLE, GREEDY, SAMPLE_BUGGY) with the per-row statistics
    of ``row_stats_batch`` on these logits (at T; at 1 for GREEDY) supplied instead of
    recomputed.  The per-row fields of the result are None."""
    B, k1, V = logits.shape
    k = k1 - 1
    lg, dt = _logits_arg(logits, dtype)
    greedy = mode == GREEDY
    qq = None if greedy else np.ascontiguousarray(q, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.int32)
    uu = None if greedy else np.ascontiguousarray(ua, dtype=np.float32)
    rr = None if greedy else np.ascontiguousarray(ur, dtype=np.float32)
    r = BatchResult(out=np.zeros((B, k1), np.int32), n=np.zeros(B, np.int32), row_m=None,
                    row_S=None, row_argmax=None, row_px=None, row_qx=None,
                    thr=np.zeros((B, k)), draw_lo=np.zeros(B), draw_hi=np.zeros(B),
                    flags=np.zeros(B, np.int32))
    c = lambda a: np.ascontiguousarray(a)
    m, S, am, bad = c(stats.m), c(stats.S), c(stats.argmax), c(stats.bad)
    rc = _load().orc_verify_batch_stats(
        int(mode), _ptr(lg), dt, _ptr(qq), _ptr(x), _ptr(uu), _ptr(rr), float(T), B, k, V,
        _ptr(m), _ptr(S), _ptr(am), _ptr(bad), _ptr(r.out), _ptr(r.n), _ptr(r.thr),
        _ptr(r.draw_lo), _ptr(r.draw_hi), _ptr(r.flags), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r


@dataclass
class Comparison:
    rows: int
    sequences: int
    mismatched_sequences: int
    near_threshold: int
    hard: int
    hard_detail: list


def compare_outputs(mode: str, ua, ur, out, n, ref: BatchResult, tol_u: float) -> Comparison:
    """Integer outputs of a verify (out [B, k+1], n [B]) against the oracle's.

    Greedy outputs must be equal.  In sampled mode a sequence that differs is a
    near-threshold case when its first differing decision had its uniform
    within tol_u of the oracle's threshold: min(1, P/Q) for an accept test (at
    the first position where the two accepted lengths differ), a bin boundary
    C_{t-1}/C_tot or C_t/C_tot for the draw; anything else is a hard mismatch.
    """
    B, k1 = out.shape
    near = hard = mism = 0
    detail = []
    for b in np.flatnonzero((n != ref.n) | np.any(out != ref.out, axis=1)):
        mism += 1
        if mode == "greedy" or n[b] < 0 or ref.n[b] < 0:
            hard += 1
            detail.append((int(b), "greedy/invalid", int(n[b]), int(ref.n[b])))
            continue
        if n[b] != ref.n[b]:
            i = int(min(n[b], ref.n[b]))
            gap = abs(float(ua[b, i]) - float(ref.thr[b, i]))
            kind = "accept"
        else:
            u = float(ur[b])
            gap = min(abs(u - ref.draw_lo[b]), abs(u - ref.draw_hi[b]))
            kind = "draw"
        if gap < tol_u:
            near += 1
        else:
            hard += 1
            detail.append((int(b), kind, gap))
    return Comparison(B * k1, B, mism, near, hard, detail[:10])


def ngram_draft(history, lengths, k: int, n_min: int, n_max: int):
    """N-gram drafter over padded histories [B, Lmax] int32 with lengths [B]:
    returns (draft [B, k] int32, -1 padded; num [B] int32)."""
    history = np.ascontiguousarray(history, dtype=np.int32)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    B, Lmax = history.shape
    draft = np.zeros((B, k), np.int32)
    num = np.zeros(B, np.int32)
    rc = _load().orc_ngram_draft(_ptr(history), _ptr(lengths), B, Lmax, int(k), int(n_min),
                                 int(n_max), _ptr(draft), _ptr(num))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return draft, num


@dataclass
class TreeResult:
    out: np.ndarray         # [N] or [B, N] accepted tokens, the emitted token, -1 after
    nodes: np.ndarray       # [N] or [B, N] accepted node indices, -1 after
    n: np.ndarray           # accepted count(s), -1 for an invalid sequence
    thr: np.ndarray         # min(1, r(x)/q(x)) of each tested child, NaN elsewhere
    draw_lo: np.ndarray
    draw_hi: np.ndarray
    flags: np.ndarray
    row_m: np.ndarray = None       # [B, N] (batch form)
    row_argmax: np.ndarray = None  # [B, N] (batch form)


def tree_seq(mode, logits, q, tok, par, ua, ur, T) -> TreeResult:
    """One sequence's tree walk with float64 inputs: logits [N, V], q [N, V]
    (sampled), tok / par [N], ua [N], ur."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    N, V = logits.shape
    qq = None if q is None else np.ascontiguousarray(q, dtype=np.float64)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    par = np.ascontiguousarray(par, dtype=np.int32)
    uu = None if ua is None else np.ascontiguousarray(ua, dtype=np.float64)
    out = np.zeros(N, np.int32)
    nodes = np.zeros(N, np.int32)
    n = np.zeros(1, np.int32)
    thr = np.zeros(N)
    lo, hi = np.zeros(1), np.zeros(1)
    fl = np.zeros(1, np.int32)
    _load().orc_tree_seq(int(mode), _ptr(logits), _ptr(qq), _ptr(tok), _ptr(par), _ptr(uu),
                         float(0.0 if ur is None else ur), float(T), N, V, _ptr(out),
                         _ptr(nodes), _ptr(n), _ptr(thr), _ptr(lo), _ptr(hi), _ptr(fl))
    return TreeResult(out, nodes, int(n[0]), thr, float(lo[0]), float(hi[0]), int(fl[0]))


def tree_batch(mode, logits, dtype: str, q, tok, par, ua, ur, T, nthreads: int = 0):
    """Batch tree walk over inputs in the device layouts: logits [B, N, V] (uint16
    bf16 bit patterns or float32), q [B, N, V] float32 (sampled), tok / par
    [B, N] int32, ua [B, N] float32, ur [B] float32."""
    B, N, V = logits.shape
    if dtype == "bf16":
        logits = np.ascontiguousarray(logits, dtype=np.uint16)
        dt = 0
    elif dtype == "f32":
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        dt = 1
    else:
        raise ValueError(dtype)
    greedy = mode == GREEDY
    qq = None if greedy else np.ascontiguousarray(q, dtype=np.float32)
    uu = None if greedy else np.ascontiguousarray(ua, dtype=np.float32)
    rr = None if greedy else np.ascontiguousarray(ur, dtype=np.float32)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    par = np.ascontiguousarray(par, dtype=np.int32)
    r = TreeResult(out=np.zeros((B, N), np.int32), nodes=np.zeros((B, N), np.int32),
                   n=np.zeros(B, np.int32), thr=np.zeros((B, N)), draw_lo=np.zeros(B),
                   draw_hi=np.zeros(B), flags=np.zeros(B, np.int32),
                   row_m=np.zeros((B, N)), row_argmax=np.zeros((B, N), np.int32))
    rc = _load().orc_tree_batch(
        int(mode), _ptr(logits), dt, _ptr(qq), _ptr(tok), _ptr(par), _ptr(uu), _ptr(rr),
        float(T), B, N, V, _ptr(r.out), _ptr(r.nodes), _ptr(r.n), _ptr(r.row_m),
        _ptr(r.row_argmax), _ptr(r.thr), _ptr(r.draw_lo), _ptr(r.draw_hi), _ptr(r.flags),
        int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return r
