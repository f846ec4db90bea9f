"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Element by element on the same seeded inputs: greedy outputs bit-exact, sampled
integer outputs equal up to counted near-threshold decisions, row statistics to
1e-5 relative.  Shapes span several tiles, ragged tails, odd V (unaligned rows),
the five named workloads at full size, and the degenerate cases.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import Guarded, compare_outputs, compare_stats, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _gen(**kw):
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    return make_inputs(**kw)


SMALL = [
    # (B, k, V, dtype, T, kind)
    (3, 1, 1, "f32", 1.0, "gauss"),
    (5, 2, 2, "bf16", 0.7, "gauss"),
    (4, 3, 3, "f32", 1.3, "gauss"),
    (16, 4, 5, "bf16", 1.0, "gauss"),
    (16, 2, 7, "f32", 0.9, "gauss"),
    (32, 5, 33, "bf16", 1.0, "zipf"),
    (64, 4, 100, "f32", 0.8, "zipf"),
    (64, 8, 1000, "bf16", 1.0, "zipf"),
    (48, 3, 4099, "f32", 0.7, "zipf"),
    (40, 5, 4099, "bf16", 1.1, "zipf"),
    (9, 2, 40000, "bf16", 0.8, "zipf"),
    (7, 6, 65537, "f32", 1.0, "zipf"),
    (2, 3, 300001, "bf16", 1.0, "zipf"),   # beyond the shared-memory slice: recompute path
]


@pytest.fixture(params=[(1, 0, 0), (1, 2, 0), (2, 0, 0), (3, 0, 0), (3, 2, 0), (3, 0, 4)],
                ids=["two_kernel", "two_kernel_cluster_draw", "fused", "skip", "skip_cluster_draw",
                     "skip_rows_in_4"])
def path(request):
    """Run a test once through each one-call path: the per-call options that
    force it (passed as run_gpu's `tuning`).  The two-kernel and row-skipping
    paths draw with the split draw (slices on separate CTAs; automatic), or
    with one cluster per sequence under draw_mode 2; the row-skipping stream
    also cuts each row into rows_split CTAs merged through the workspace."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    p, dm, rsplit = request.param
    return sv.Tuning(path=p, draw_mode=dm, rows_split=rsplit)


@pytest.mark.parametrize("B,k,V,dtype,T,kind", SMALL)
def test_sampled_small(B, k, V, dtype, T, kind, path):
    inp = _gen(mode="sample", B=B, k=k, V=V, dtype=dtype, T=T, kind=kind, seed=B * 7 + V)
    out, n, stats, (st, bits, ndeg) = run_gpu(inp, tuning=path)
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0, rep.hard_detail
    assert rep.near_threshold <= 1
    assert st == 0 and (bits & 0xF) == 0
    compare_stats(inp, stats, ref, n)


@pytest.mark.parametrize("B,k,V,dtype,T,kind", SMALL)
def test_greedy_small(B, k, V, dtype, T, kind, path):
    inp = _gen(mode="greedy", B=B, k=k, V=V, dtype=dtype, kind=kind, p_argmax=0.7,
               seed=B * 11 + V)
    out, n, stats, (st, bits, _) = run_gpu(inp, tuning=path)
    ref = run_oracle(inp)
    assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    assert st == 0 and (bits & 0xF) == 0
    compare_stats(inp, stats, ref, n)


def test_two_stage_equals_one_call(path):
    for mode in ("sample", "greedy"):
        inp = _gen(mode=mode, B=24, k=4, V=5000, dtype="bf16", T=0.9, kind="zipf", seed=5)
        dev = to_device(inp)
        a = run_gpu(inp, dev, tuning=path)
        b = run_gpu(inp, dev, two_stage=True, tuning=path)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_workload_fused_path(name):
    """The fused kernel on workloads the automatic dispatch sends elsewhere."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import workload
    inp = workload(name, seed=11)
    out, n, stats, (st, bits, _) = run_gpu(inp, tuning=sv.Tuning(path=sv.PATH_FUSED))
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0 and rep.near_threshold <= 1, rep.hard_detail
    compare_stats(inp, stats, ref, n)


@pytest.mark.parametrize("mode", ["sample", "greedy"])
@pytest.mark.parametrize("rows_split", [0, 4], ids=["one_cta_per_row", "rows_in_4"])
def test_skip_path_skips_rows_and_matches(mode, rows_split):
    """The row-skipping path on a batch of many waves of rows: later rows of a
    sequence that has already stopped are not read (their statistics come back
    unset), and every output still equals the oracle's; with each row cut into
    four CTAs merged through the workspace too."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    inp = _gen(mode=mode, B=2048, k=6, V=2000, dtype="bf16", T=0.9, kind="zipf", p_argmax=0.6,
               seed=77)
    out, n, stats, (st, bits, _) = run_gpu(inp, tuning=sv.Tuning(path=sv.PATH_SKIP,
                                                                 rows_split=rows_split))
    ref = run_oracle(inp)
    if mode == "greedy":
        assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    else:
        rep = compare_outputs(inp, out, n, ref)
        assert rep.hard == 0 and rep.near_threshold <= 2, rep.hard_detail
    assert st == 0 and (bits & 0xF) == 0
    compare_stats(inp, stats, ref, n)
    argmax = stats["argmax"].reshape(inp.B, inp.k + 1)
    skipped = argmax < 0
    # never a row at or before the decision row
    assert not any(skipped[b, : n[b] + 1].any() for b in range(inp.B))
    assert skipped.sum() > 0


@pytest.mark.parametrize("name", ["c4"])
def test_workload_fused_path_large(name):
    """The fused per-sequence kernel on the large-batch workload."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import workload
    inp = workload(name, seed=12)
    out, n, stats, (st, bits, _) = run_gpu(inp, tuning=sv.Tuning(path=sv.PATH_FUSED))
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0 and rep.near_threshold <= 1, rep.hard_detail


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_workload_full_size(name):
    """The five named workloads at full size, every sequence compared."""
    from speculative_decoding_verification_18_gb300.inputs import workload
    inp = workload(name)
    out, n, stats, (st, bits, _) = run_gpu(inp)
    ref = run_oracle(inp)
    if inp.mode == "greedy":
        assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    else:
        rep = compare_outputs(inp, out, n, ref)
        assert rep.hard == 0, rep.hard_detail
        assert rep.near_threshold <= max(1, rep.rows // 100000)
    assert st == 0 and (bits & 0xF) == 0
    compare_stats(inp, stats, ref, n)


def test_config1_shape_many_sequences():
    """Config-1-shaped inputs (V=32, k=4, N(0, 2^2) logits, T=1) over 20000 sequences."""
    inp = _gen(mode="sample", B=20000, k=4, V=32, dtype="f32", T=1.0, kind="gauss", scale=2.0,
               draft_sigma=0.5, seed=99)
    out, n, stats, _ = run_gpu(inp)
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0, rep.hard_detail
    assert rep.near_threshold <= 2
    compare_stats(inp, stats, ref, n)


def test_mismatch_rate_two_hundred_thousand_rows():
    """Near-threshold mismatches stay below 1e-5 of rows over 2e5 rows of Zipf bf16."""
    rows = near = 0
    for s in range(20):
        inp = _gen(mode="sample", B=2000, k=4, V=4096, dtype="bf16", T=0.8, kind="zipf",
                   draft_sigma=0.7, seed=1000 + s)
        out, n, _, _ = run_gpu(inp)
        ref = run_oracle(inp)
        rep = compare_outputs(inp, out, n, ref)
        assert rep.hard == 0, rep.hard_detail
        rows += rep.rows
        near += rep.near_threshold
    assert rows >= 200000
    assert near <= 2  # < 1e-5 of rows


def test_ffexp_accuracy():
    """The draw's float-float exponential against float64 exp.  The argument
    (l - m)/T is carried to ~2^-47 relative, so the bound grows with |z|:
    relative error <= 2e-14 * (1 + |z|) (about 2^-45.5 per unit of |z|)."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    g = np.random.default_rng(3)
    for T in (1.0, 0.7, 0.8, 1.3):
        m = np.float32(5.25)
        l = (m - g.uniform(0, 44 * T, 200000)).astype(np.float32)
        l[:5] = [m, m - 1e-7, m - 0.5, np.float32(-1e-30), m - 44 * T]
        e = sv.debug_ffexp(torch.from_numpy(l).cuda(), float(m), T).cpu().numpy()
        z = (l.astype(np.float64) - np.float64(m)) / np.float64(np.float32(T))
        ref = np.exp(z)
        ok = z > -43.9
        rel = np.abs(e[ok] - ref[ok]) / ref[ok]
        bound = 2e-14 * (1.0 + np.abs(z[ok]))
        assert (rel <= bound).all(), (rel / bound).max()
        assert (e[~ok] >= 0).all() and (e[~ok] < 1e-18).all()


def test_ex2_approx_error_within_the_fast_draw_bound():
    """The fast draw's error bound takes ex2.approx.ftz.f32 to be within 1.75e-7
    of 2^a (relative); measured exhaustively over every float in [-126, 0]
    against the float-float exponential it must be no worse (GB300: 1.715e-7)."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    worst = sv.debug_ex2_error(-126.0, 0.0)
    assert 0.0 < worst <= 1.75e-7, worst


@pytest.mark.parametrize("name,path,draw_mode", [
    ("c3", 2, 0), ("c3", 1, 1), ("c3", 1, 2), ("c4", 0, 1), ("c4", 0, 2), ("c5", 0, 1),
    ("c5", 0, 2)], ids=["c3-fused", "c3-split", "c3-cluster", "c4-split", "c4-cluster",
                        "c5-split", "c5-cluster"])
def test_workload_precise_draw_only(name, path, draw_mode):
    """Every draw through the float-float pass (the fast pass switched off), in
    the fused kernel, the split precise draw and the cluster draw."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import workload
    inp = workload(name, seed=77)
    out, n, stats, (st, bits, _) = run_gpu(
        inp, tuning=sv.Tuning(force_precise=1, path=path, draw_mode=draw_mode))
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0, rep.hard_detail
    assert rep.near_threshold <= max(1, rep.rows // 100000)
    assert bits & sv.SV_DEV_PRECISE and st == 0


def test_both_draw_passes_occur():
    """On the long-tailed fp32 workload some draws certify in the fast pass and
    some need the precise one (counted per sequence)."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    inp = make_inputs(mode="sample", B=256, k=3, V=151936, dtype="f32", T=1.0, kind="zipf",
                      slope=1.0, noise=1.5, draft_sigma=1.0, seed=31)
    out, n, stats, (st, bits, _) = run_gpu(inp)
    assert bits & sv.SV_DEV_PRECISE
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0, rep.hard_detail


def test_graph_capture_replay():
    """The one-call form captures into a CUDA graph and replays identically."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    inp = _gen(mode="sample", B=16, k=5, V=20000, dtype="bf16", T=0.8, kind="zipf", seed=8)
    dev = to_device(inp)
    gd = Guarded()
    ws = gd.workspace(inp.B, inp.k, inp.V, torch.bfloat16)
    out = gd.empty((inp.B, inp.k + 1), torch.int32)
    n = gd.empty(inp.B, torch.int32)
    sv.spec_verify_sample(dev["logits"], dev["q"], dev["x"], dev["ua"], dev["ur"], inp.T, out, n,
                          ws)  # first call outside capture (device set-up)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sv.spec_verify_sample(dev["logits"], dev["q"], dev["x"], dev["ua"], dev["ur"], inp.T,
                                  out, n, ws)
    out.fill_(-9)
    g.replay()
    torch.cuda.synchronize()
    gd.check()
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out.cpu().numpy(), n.cpu().numpy(), ref)
    assert rep.hard == 0 and rep.near_threshold == 0


# ---------------------------------------------------------------- edge cases

def _single(logits, q, x, ua, ur, T, dtype="f32", tuning=None):
    """Run one hand-made batch on both sides."""
    from speculative_decoding_verification_18_gb300.inputs import VerifyInputs, bf16_bits
    logits = np.asarray(logits, np.float32)
    B, k1, V = logits.shape
    lg = bf16_bits(logits) if dtype == "bf16" else logits
    inp = VerifyInputs("sample", dtype, B, k1 - 1, V, T, lg, np.asarray(q, np.float32),
                       np.asarray(x, np.int32), np.asarray(ua, np.float32),
                       np.asarray(ur, np.float32))
    out, n, stats, st = run_gpu(inp, tuning=tuning)
    ref = run_oracle(inp)
    return inp, out, n, st, ref


def test_invalid_data_marks_sequence(path):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    V, k = 6, 3
    base = np.log(np.array([0.1, 0.2, 0.3, 0.1, 0.2, 0.1]))
    logits = np.tile(base, (6, k + 1, 1))
    q = np.tile(np.array([0.3, 0.1, 0.2, 0.2, 0.1, 0.1]), (6, k, 1))
    x = np.array([[2, 2, 2]] * 6)
    ua = np.full((6, k), 0.5)
    ur = np.full(6, 0.5)
    x[1, 0] = 6                 # token out of range
    logits[2, 0, 3] = np.nan     # NaN in a reached row
    logits[3, 1, :] = -np.inf    # all -inf reached row
    ua[4, 0] = 1.0               # uniform out of range
    q[5, 0, 2] = np.nan          # q(x) NaN
    inp, out, n, (st, bits, _), ref = _single(logits, q, x, ua, ur, 1.0, tuning=path)
    assert list(ref.n) == [3, -1, -1, -1, -1, -1]
    assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    assert st == sv.SV_ERR_DATA
    want = (sv.SV_DEV_BAD_TOKEN | sv.SV_DEV_BAD_ROW | sv.SV_DEV_BAD_UNIFORM | sv.SV_DEV_BAD_Q)
    assert bits & want == want


def test_bad_row_after_rejection_is_not_read():
    V, k = 5, 2
    logits = np.tile(np.log(np.array([0.1, 0.2, 0.3, 0.15, 0.25])), (1, k + 1, 1))
    logits[0, 2, 1] = np.nan
    q = np.tile(np.array([0.0, 0.5, 0.1, 0.2, 0.2]), (1, k, 1))
    inp, out, n, (st, bits, _), ref = _single(logits, q, [[1, 0]], [[0.9, 0.1]], [0.3], 1.0)
    assert n[0] == 0 and ref.n[0] == 0 and out[0, 0] == ref.out[0, 0]
    assert st == 0


def test_accept_rules_and_degenerate_residual(path):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    V, k = 5, 2
    logits = np.tile(np.log(np.array([0.1, 0.2, 0.3, 0.15, 0.25])), (3, k + 1, 1))
    q = np.tile(np.array([0.0, 0.5, 0.1, 0.2, 0.2]), (3, k, 1))
    x = np.array([[0, 2], [1, 2], [1, 0]])
    ua = np.array([[0.999, 0.999], [0.2 / 0.5 + 1e-3, 0.0], [0.9, 0.1]])
    q[2] = np.array([0.2, 0.4, 0.31, 0.16, 0.26])  # q > p everywhere: zero residual mass
    ur = np.array([0.3, 0.3, 0.05])
    inp, out, n, (st, bits, ndeg), ref = _single(logits, q, x, ua, ur, 1.0, tuning=path)
    assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    assert n[0] == 2 and n[1] == 0 and n[2] == 0
    assert ref.flags[2] & oracle.F_DEGENERATE
    assert bits & sv.SV_DEV_DEGENERATE and ndeg == 1 and st == sv.SV_OK


def test_zero_weight_bins_never_drawn():
    """Rejections whose residual is zero on half the vocabulary, swept over u."""
    g = np.random.default_rng(4)
    V, k, B = 64, 1, 4096
    l = g.normal(0, 1, V)
    p = np.exp(l - l.max())
    p /= p.sum()
    qrow = np.where(np.arange(V) % 2 == 0, p * 1.5, p * 0.5)
    qrow /= qrow.sum()
    xr = int(np.argmax(qrow / p))
    logits = np.tile(l, (B, k + 1, 1))
    q = np.tile(qrow, (B, k, 1))
    x = np.full((B, k), xr)
    ua = np.full((B, k), 0.999999)
    ur = (np.arange(B) + 0.5) / B
    inp, out, n, _, ref = _single(logits, q, x, ua, ur, 1.0)
    assert (n == 0).all()
    w = np.maximum(p - qrow.astype(np.float32).astype(np.float64), 0)
    assert (w[out[:, 0]] > 0).all()
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0


def test_v_equals_one_and_empty_batch():
    from speculative_decoding_verification_18_gb300 import specverify as sv
    inp, out, n, (st, _, _), ref = _single(np.zeros((2, 3, 1)), np.ones((2, 2, 1)),
                                           [[0, 0], [0, 0]], [[0.5, 0.5]] * 2, [0.5, 0.99], 1.0)
    assert (n == 2).all() and (out == 0).all()
    ws = sv.workspace(0, 3, 10)
    e = torch.empty((0, 4, 10), dtype=torch.float32, device="cuda")
    sv.spec_verify_sample(e, torch.empty((0, 3, 10), device="cuda"),
                          torch.empty((0, 3), dtype=torch.int32, device="cuda"),
                          torch.empty((0, 3), device="cuda"), torch.empty(0, device="cuda"), 1.0,
                          torch.empty((0, 4), dtype=torch.int32, device="cuda"),
                          torch.empty(0, dtype=torch.int32, device="cuda"), ws)


def test_bf16_ties_lowest_index(path):
    """Many exact ties in bf16: argmax and greedy outputs pick the lowest index."""
    B, k, V = 32, 3, 3000
    g = np.random.default_rng(1)
    vals = g.integers(-4, 4, (B, k + 1, V)).astype(np.float32)
    from speculative_decoding_verification_18_gb300.inputs import VerifyInputs, bf16_bits
    am = vals.argmax(axis=2)
    x = np.where(g.random((B, k)) < 0.5, am[:, :k], 0).astype(np.int32)
    inp = VerifyInputs("greedy", "bf16", B, k, V, 1.0, bf16_bits(vals), None, x, None, None)
    out, n, stats, _ = run_gpu(inp, tuning=path)
    ref = run_oracle(inp)
    assert np.array_equal(out, ref.out) and np.array_equal(n, ref.n)
    # every row the GPU read (the row-skipping path may leave rows past the
    # decision row unread: argmax -1) has the lowest index of its maximum
    got = stats["argmax"].reshape(B, k + 1)
    read = got >= 0
    assert all(read[b, : n[b] + 1].all() for b in range(B))
    assert np.array_equal(got[read], am[read])


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_maximum_k_and_vocabulary(mode, path):
    """The largest sizes the ABI accepts: k = 64 drafts and V = 2^21 tokens
    (one sequence, bf16), and k = 64 over a batch, through every path."""
    for B, V in ((1, 1 << 21), (24, 3000)):
        inp = _gen(mode=mode, B=B, k=64, V=V, dtype="bf16", T=1.0, kind="zipf",
                   p_argmax=0.97, draft_sigma=0.05, seed=V + B)
        out, n, stats, (st, bits, _) = run_gpu(inp, tuning=path)
        ref = run_oracle(inp)
        rep = compare_outputs(inp, out, n, ref)
        assert rep.hard == 0, rep.hard_detail
        assert st == 0
