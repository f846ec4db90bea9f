"""GPU parity of the flat greedy row stream against the float64 oracle.

Greedy verification needs only each row's argmax ("Decodificação especulativa
explicada", the greedy special case: accept while the draft equals the target's
argmax).  When a greedy batch has about as many rows as the GPU holds CTAs, the
row stream cuts the whole logits tensor into one equal range per resident CTA;
a range may cover parts of up to four rows and a row may be spread over up to
four ranges, and the finish kernel merges the partial keys.  These tests pick
shapes where that happens (checked with the introspection hook) and require
bit-exact outputs and row statistics, with the flat stream on and off, including
ties across range boundaries, NaN / infinite rows and bad draft tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import Guarded, compare_outputs, compare_stats, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(params=[0, 1], ids=["flat", "per_row"])
def flat_off(request):
    """0: the automatic choice (the flat stream for these shapes); 1: the per-row
    stream, through the per-call option."""
    return request.param


def _tuning(off):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    return sv.Tuning(flat_off=1) if off else None


def _greedy(B, k, V, dtype, seed, p_argmax=0.7):
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    return make_inputs(mode="greedy", B=B, k=k, V=V, dtype=dtype, T=1.0, kind="zipf",
                       p_argmax=p_argmax, seed=seed)


def _flat_ctas(inp):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    return sv.debug_flat_ctas(inp.B, inp.k, inp.V, inp.dtype)


def _check(inp, off=0):
    out, n, stats, (st, bits, _) = run_gpu(inp, tuning=_tuning(off))
    ref = run_oracle(inp)
    rep = compare_outputs(inp, out, n, ref)
    assert rep.hard == 0 and rep.mismatched_sequences == 0, rep.hard_detail
    compare_stats(inp, stats, ref, n)
    return out, n, stats, st, bits, ref


FLAT_SHAPES = [
    # (B, k, V, dtype): ranges of several rows, of about one row, of parts of rows
    (64, 4, 32000, "bf16"),   # the greedy workload's shape
    (64, 4, 100, "f32"),      # 25-vector rows: each range covers up to four rows
    (40, 3, 8192, "bf16"),
    (100, 2, 4096, "f32"),
    (60, 6, 1000, "bf16"),
    (25, 3, 65536, "f32"),    # ranges of about a third of a row
]


@pytest.mark.parametrize("B,k,V,dtype", FLAT_SHAPES)
def test_flat_matches_oracle(B, k, V, dtype, flat_off):
    inp = _greedy(B, k, V, dtype, seed=B + k + V)
    if not flat_off:
        assert _flat_ctas(inp) > 0, "shape expected on the flat stream"
    _check(inp, flat_off)


def test_flat_is_taken_by_the_greedy_workload():
    from speculative_decoding_verification_18_gb300.inputs import workload
    inp = workload("c2")
    P = _flat_ctas(inp)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms <= P <= 2 * sms


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_flat_ties_across_ranges(dtype, flat_off):
    """Rows of equal values, and maxima repeated at both ends of every row: the
    lowest index must win even when the copies lie in different CTAs' ranges."""
    from speculative_decoding_verification_18_gb300.inputs import VerifyInputs, bf16_bits
    B, k, V = 64, 4, 2048
    g = np.random.default_rng(5)
    vals = g.integers(-3, 3, (B, k + 1, V)).astype(np.float32)
    vals[::3] = 1.5                          # whole sequences of constant rows
    vals[1::3, :, 0] = 9.0                   # the maximum at both ends of the row
    vals[1::3, :, V - 1] = 9.0
    vals[2::3, :, V // 2] = 7.0              # mid-row maximum, repeated near the end
    vals[2::3, :, V - 3] = 7.0
    am = vals.argmax(axis=2)
    x = np.where(g.random((B, k)) < 0.6, am[:, :k], (am[:, :k] + 1) % V).astype(np.int32)
    logits = bf16_bits(vals) if dtype == "bf16" else vals
    inp = VerifyInputs("greedy", dtype, B, k, V, 1.0, logits, None, x, None, None)
    if not flat_off:
        assert _flat_ctas(inp) > 0
    out, n, stats, st, bits, ref = _check(inp, flat_off)
    assert np.array_equal(stats["argmax"], am)


def test_flat_invalid_rows_and_tokens(flat_off):
    """NaN, all -inf and +inf rows mark their sequence bad when the scan reaches
    them; an out-of-range draft token marks it too; rows past the stop do not."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    inp = _greedy(64, 4, 4096, "f32", seed=17, p_argmax=1.0)
    lg = inp.logits
    lg[1, 0, 5] = np.nan                      # NaN in row 0
    lg[2, 2, :] = -np.inf                     # all -inf row 2 (reached: p_argmax = 1)
    lg[3, 1, 4000] = np.inf                   # +inf in row 1
    inp.x[4, 1] = 4096                        # token out of range
    inp.x[5, 0] = -1
    inp.x[6, 0] = (inp.x[6, 0] + 1) % 4096    # rejected at 0 ...
    lg[6, 3, 7] = np.nan                      # ... so this NaN row is never judged
    if not flat_off:
        assert _flat_ctas(inp) > 0
    out, n, stats, (st, bits, _) = run_gpu(inp, tuning=_tuning(flat_off))
    ref = run_oracle(inp)
    assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    assert list(n[1:7]) == [-1, -1, -1, -1, -1, 0]
    assert st == sv.SV_ERR_DATA
    want = sv.SV_DEV_BAD_TOKEN | sv.SV_DEV_BAD_ROW
    assert bits & want == want


def test_flat_two_stage_and_graph_replay():
    """spec_verify_rows + spec_verify_finish equal the one call, and a captured
    graph of the flat path replays to the same outputs."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    inp = _greedy(64, 4, 32000, "bf16", seed=3)
    assert _flat_ctas(inp) > 0
    out1, n1, _, _ = run_gpu(inp)
    out2, n2, _, _ = run_gpu(inp, two_stage=True)
    assert np.array_equal(out1, out2) and np.array_equal(n1, n2)
    lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).cuda()
    x = torch.from_numpy(inp.x).cuda()
    gd = Guarded()
    out = gd.empty((64, 5), torch.int32, fill=-7)
    n = gd.empty((64,), torch.int32, fill=-7)
    ws = gd.workspace(64, 4, 32000, torch.bfloat16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sv.spec_verify_greedy(lg, x, out, n, ws)
        torch.cuda.synchronize()
        out.fill_(-7)
        n.fill_(-7)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            sv.spec_verify_greedy(lg, x, out, n, ws)
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    gd.check()
    assert np.array_equal(out.cpu().numpy(), out1) and np.array_equal(n.cpu().numpy(), n1)


def test_workspace_reused_across_paths():
    """One workspace through the flat greedy stream, a sampled verify, the
    per-row greedy stream, a tree verify and the flat stream again: every
    call's outputs equal the oracle's (each call rewrites the layout word the
    finish kernels read)."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs, make_tree_inputs
    B, k, V = 64, 4, 8192
    g_in = make_inputs(mode="greedy", B=B, k=k, V=V, dtype="bf16", kind="zipf", seed=41)
    s_in = make_inputs(mode="sample", B=B, k=k, V=V, dtype="bf16", T=0.9, kind="zipf",
                       draft_sigma=0.4, seed=42)
    t_in = make_tree_inputs(mode="greedy", B=B, N=k + 1, V=V, dtype="bf16", branching=(2,),
                            seed=43)
    gd = Guarded()
    ws = gd.workspace(B, k, V, torch.bfloat16)
    assert _flat_ctas(g_in) > 0
    for step, off in enumerate([0, None, 1, "tree", 0]):
        if off == "tree":
            lg = torch.from_numpy(t_in.logits.view(np.int16)).view(torch.bfloat16).cuda()
            out = gd.empty((B, k + 1), torch.int32)
            nodes = gd.empty((B, k + 1), torch.int32)
            n = gd.empty(B, torch.int32)
            sv.spec_verify_tree(sv.SV_MODE_GREEDY, lg, None, torch.from_numpy(t_in.tok).cuda(),
                                torch.from_numpy(t_in.par).cuda(), None, None, 1.0, out, nodes,
                                n, ws)
            torch.cuda.synchronize()
            gd.check()
            ref = oracle.tree_batch(oracle.GREEDY, t_in.logits, "bf16", None, t_in.tok, t_in.par,
                                    None, None, 1.0)
            assert np.array_equal(out.cpu().numpy(), ref.out), step
            continue
        inp = s_in if off is None else g_in
        out, n, stats, _ = run_gpu(inp, ws=ws, tuning=_tuning(off))
        ref = run_oracle(inp)
        rep = compare_outputs(inp, out, n, ref)
        assert rep.hard == 0, (step, rep.hard_detail)


def test_flat_finish_twice_and_stats_before_finish():
    """After one flat spec_verify_rows, spec_verify_row_stats (which merges the
    partial keys on the host) and two spec_verify_finish calls in a row all agree
    with the oracle: the finish merges the keys into copies of its own and leaves
    them in the workspace, so it can run again on the same row stream output."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    for B, k, V, dtype in ((64, 4, 32000, "bf16"), (40, 3, 12000, "f32")):
        inp = _greedy(B, k, V, dtype, seed=B + V)
        assert _flat_ctas(inp) > 0
        ref = run_oracle(inp)
        if dtype == "bf16":
            lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).cuda()
        else:
            lg = torch.from_numpy(inp.logits).cuda()
        x = torch.from_numpy(inp.x).cuda()
        gd = Guarded()
        ws = gd.workspace(B, k, V, lg.dtype)
        sv.spec_verify_rows(sv.SV_MODE_GREEDY, lg, None, x, 1.0, ws)
        stats = sv.spec_verify_row_stats(ws, B, k)
        assert np.array_equal(stats["argmax"], ref.row_argmax)
        assert np.array_equal(stats["m"].astype(np.float64), ref.row_m)
        for rep in range(2):
            out = gd.empty((B, k + 1), torch.int32, fill=-7)
            n = gd.empty(B, torch.int32, fill=-7)
            sv.spec_verify_finish(sv.SV_MODE_GREEDY, lg, None, x, None, None, 1.0, out, n, ws)
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy(), ref.out), rep
            assert np.array_equal(n.cpu().numpy(), ref.n), rep
        stats = sv.spec_verify_row_stats(ws, B, k)
        assert np.array_equal(stats["argmax"], ref.row_argmax)
        gd.check()
