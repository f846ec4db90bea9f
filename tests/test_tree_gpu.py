"""GPU parity of tree verification (spec_verify_tree) against the oracle.

Several drafted continuations checked at once ("Decodificação especulativa
explicada", §"A família de rascunhos", Medusa's tree attention).  Greedy outputs
must equal the oracle's bit for bit; sampled outputs too, except a sequence
whose first differing decision had its uniform within 1e-5 of the oracle's
threshold (an accept test) or bin edge (the final draw), counted.  Also: trees
that are chains equal the chain entry points, malformed trees and bad data are
flagged, and on the page's toy the first emitted token follows p.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import Guarded

pytestmark = pytest.mark.gpu

TOL_U = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_tree(t):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    B, N, V = t.B, t.N, t.V
    if t.dtype == "bf16":
        lg = torch.from_numpy(t.logits.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        lg = torch.from_numpy(t.logits).cuda()
    sampled = t.mode == "sample"
    q = torch.from_numpy(t.q).cuda() if sampled else None
    ua = torch.from_numpy(t.ua).cuda() if sampled else None
    ur = torch.from_numpy(t.ur).cuda() if sampled else None
    tok = torch.from_numpy(t.tok).cuda()
    par = torch.from_numpy(t.par).cuda()
    g = Guarded()
    out = g.empty((B, N), torch.int32, fill=-7)
    nodes = g.empty((B, N), torch.int32, fill=-7)
    n = g.empty((B,), torch.int32, fill=-7)
    ws = g.workspace(B, N - 1, V, lg.dtype)
    mode = sv.SV_MODE_SAMPLE if sampled else sv.SV_MODE_GREEDY
    sv.spec_verify_tree(mode, lg, q, tok, par, ua, ur, t.T, out, nodes, n, ws)
    torch.cuda.synchronize()
    g.check()
    st, bits, _ = sv.spec_verify_read_status(ws)
    return out.cpu().numpy(), nodes.cpu().numpy(), n.cpu().numpy(), st, bits, ws


def run_oracle(t):
    mode = oracle.SAMPLE if t.mode == "sample" else oracle.GREEDY
    return oracle.tree_batch(mode, t.logits, t.dtype, t.q, t.tok, t.par, t.ua, t.ur, t.T)


def compare(t, out, nodes, n, ref):
    """(hard mismatches, near-threshold mismatches)."""
    hard, near = [], 0
    for b in np.nonzero((n != ref.n) | (out != ref.out).any(axis=1)
                        | (nodes != ref.nodes).any(axis=1))[0]:
        if t.mode == "greedy" or n[b] < 0 or ref.n[b] < 0:
            hard.append(int(b))
            continue
        gaps = [abs(float(t.ua[b, j]) - ref.thr[b, j]) for j in range(1, t.N)
                if not np.isnan(ref.thr[b, j])]
        gaps += [abs(float(t.ur[b]) - ref.draw_lo[b]), abs(float(t.ur[b]) - ref.draw_hi[b])]
        if min(gaps) < TOL_U:
            near += 1
        else:
            hard.append(int(b))
    return hard, near


CASES = [
    # (mode, B, N, V, dtype, T, branching or None for random shapes)
    ("greedy", 8, 2, 5, "f32", 1.0, (1,)),
    ("greedy", 16, 7, 33, "bf16", 1.0, None),
    ("greedy", 64, 5, 32000, "bf16", 1.0, (1,)),       # a chain: the flat stream's shape
    ("greedy", 32, 16, 4099, "f32", 1.0, (4, 2, 2)),
    ("greedy", 4, 65, 1000, "bf16", 1.0, None),
    ("sample", 8, 2, 5, "f32", 1.0, (1,)),
    ("sample", 16, 7, 33, "bf16", 0.8, None),
    ("sample", 32, 16, 4099, "f32", 1.0, (4, 2, 2)),
    ("sample", 24, 12, 32000, "bf16", 0.9, (3, 2, 1)),
    ("sample", 6, 9, 40001, "bf16", 1.2, (8,)),         # one level of 8 siblings
    ("sample", 4, 65, 1000, "f32", 1.0, None),
]


@pytest.mark.parametrize("mode,B,N,V,dtype,T,branching", CASES)
def test_tree_matches_oracle(mode, B, N, V, dtype, T, branching):
    from speculative_decoding_verification_18_gb300.inputs import make_tree_inputs
    t = make_tree_inputs(mode=mode, B=B, N=N, V=V, dtype=dtype, T=T,
                         branching=branching or (2,), random_shape=branching is None,
                         draft_sigma=0.5, seed=B * 7 + N + V)
    out, nodes, n, st, bits, ws = run_tree(t)
    ref = run_oracle(t)
    hard, near = compare(t, out, nodes, n, ref)
    assert not hard, hard[:5]
    assert near <= 1
    assert st == 0 and (bits & 0x4F) == 0
    assert (n >= 0).all()
    if mode == "greedy":  # row argmaxes of every node (the walk's records)
        from speculative_decoding_verification_18_gb300 import specverify as sv
        stats = sv.spec_verify_row_stats(ws, B, N - 1)
        assert np.array_equal(stats["argmax"], ref.row_argmax)


@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_chain_tree_equals_chain_verify(mode):
    """A chain-shaped tree gives what the chain entry points give on the same rows."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    B, k, V = 48, 4, 3000
    inp = make_inputs(mode=mode, B=B, k=k, V=V, dtype="bf16", T=0.9, kind="zipf",
                      draft_sigma=0.4, seed=31)
    lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).cuda()
    x = torch.from_numpy(inp.x).cuda()
    g = Guarded()
    out_c = g.empty((B, k + 1), torch.int32)
    n_c = g.empty(B, torch.int32)
    ws = g.workspace(B, k, V, lg.dtype)
    tok = torch.from_numpy(np.hstack([np.full((B, 1), -1, np.int32), inp.x])).cuda()
    par = torch.from_numpy(np.tile(np.r_[-1, np.arange(k)].astype(np.int32), (B, 1))).cuda()
    out_t = g.empty((B, k + 1), torch.int32)
    nodes = g.empty((B, k + 1), torch.int32)
    n_t = g.empty(B, torch.int32)
    ws_t = g.workspace(B, k, V, lg.dtype)
    if mode == "greedy":
        sv.spec_verify_greedy(lg, x, out_c, n_c, ws)
        sv.spec_verify_tree(sv.SV_MODE_GREEDY, lg, None, tok, par, None, None, 1.0, out_t,
                            nodes, n_t, ws_t)
    else:
        q = torch.from_numpy(inp.q).cuda()
        ua = torch.from_numpy(inp.ua).cuda()
        ur = torch.from_numpy(inp.ur).cuda()
        sv.spec_verify_sample(lg, q, x, ua, ur, inp.T, out_c, n_c, ws)
        qt = torch.cat([q, torch.full((B, 1, V), 0.5, device="cuda")], dim=1).contiguous()
        uat = torch.cat([torch.zeros((B, 1), device="cuda"), ua], dim=1).contiguous()
        sv.spec_verify_tree(sv.SV_MODE_SAMPLE, lg, qt, tok, par, uat, ur, inp.T, out_t, nodes,
                            n_t, ws_t)
    torch.cuda.synchronize()
    g.check()
    a_o, a_n = out_c.cpu().numpy(), n_c.cpu().numpy()
    b_o, b_n = out_t.cpu().numpy(), n_t.cpu().numpy()
    same = (a_n == b_n) & (a_o == b_o).all(axis=1)
    # the two draws compute their weights differently (certified fast pass vs
    # fp32 weights with float64 sums): allow the rare boundary case
    assert same.sum() >= B - 1, np.nonzero(~same)[0]
    nd = nodes.cpu().numpy()
    for b in range(B):
        assert list(nd[b, :b_n[b]]) == list(range(1, b_n[b] + 1))


def test_tree_invalid_data():
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_tree_inputs
    t = make_tree_inputs(mode="sample", B=8, N=7, V=300, dtype="f32", branching=(2,),
                         seed=5)
    t.ua[:] = 0.0                       # every tested child accepted
    t.par[1, 3] = 3                      # malformed tree
    t.tok[2, 1] = 300                    # token out of range at a tested child
    t.logits[3, 0, 5] = np.nan           # the root row
    t.ua[4, 1] = 1.5                     # bad uniform at a tested child
    t.ur[5] = -1.0                       # bad final uniform (reached: leaves at depth 2)
    out, nodes, n, st, bits, _ = run_tree(t)
    ref = run_oracle(t)
    assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    assert list(n[1:6]) == [-1, -1, -1, -1, -1]
    assert (out[1:6] == -1).all() and (nodes[1:6] == -1).all()
    assert st == sv.SV_ERR_DATA
    want = sv.SV_DEV_BAD_TREE | sv.SV_DEV_BAD_TOKEN | sv.SV_DEV_BAD_ROW | sv.SV_DEV_BAD_UNIFORM
    assert bits & want == want


def test_tree_first_token_follows_p():
    """The page's toy (V = 4): a root with three children drawn independently
    from Q[c], each child a leaf.  Over 300 000 sequences per context the first
    emitted token follows P[c] (chi-square)."""
    from scipy.stats import chi2
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    P, Q = toy_language()
    M, N, V = 300_000, 4, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    par = torch.tensor([-1, 0, 0, 0], dtype=torch.int32, device="cuda").expand(M, N).contiguous()
    for c in range(4):
        lnP = torch.from_numpy(np.log(P).astype(np.float32)).cuda()
        logits = lnP[c].expand(M, N, V).contiguous()
        q = torch.from_numpy(Q[c].astype(np.float32)).cuda().expand(M, N, V).contiguous()
        cq = torch.cumsum(torch.from_numpy(Q[c].astype(np.float32)).cuda(), 0)
        u = torch.rand((M, N), device="cuda", generator=g)
        tok = torch.searchsorted(cq.expand(M, V).contiguous(), (u * cq[-1]).contiguous(),
                                 right=True).clamp_(max=V - 1).to(torch.int32)
        tok[:, 0] = -1
        ua = torch.rand((M, N), device="cuda", generator=g)
        ur = torch.rand(M, device="cuda", generator=g)
        gd = Guarded()
        out = gd.empty((M, N), torch.int32)
        nodes = gd.empty((M, N), torch.int32)
        n = gd.empty(M, torch.int32)
        ws = gd.workspace(M, N - 1, V, torch.float32)
        sv.spec_verify_tree(sv.SV_MODE_SAMPLE, logits, q, tok.contiguous(), par, ua, ur, 1.0,
                            out, nodes, n, ws)
        torch.cuda.synchronize()
        gd.check()
        first = out[:, 0].cpu().numpy()
        counts = np.bincount(first, minlength=4).astype(float)
        stat = float(((counts - M * P[c]) ** 2 / (M * P[c])).sum())
        assert chi2.sf(stat, 3) > 1e-4, (c, stat, counts / M, P[c])


def test_tree_mismatch_rate_many_trees():
    """20 000 sampled trees of 8 nodes (V = 1000): no hard mismatch, and the
    near-threshold ones (fp32 weights against float64) rare."""
    from speculative_decoding_verification_18_gb300.inputs import make_tree_inputs
    t = make_tree_inputs(mode="sample", B=20000, N=8, V=1000, dtype="bf16", T=1.0,
                         branching=(3, 2), draft_sigma=0.6, seed=77)
    out, nodes, n, st, bits, _ = run_tree(t)
    ref = run_oracle(t)
    hard, near = compare(t, out, nodes, n, ref)
    assert not hard, hard[:5]
    assert near <= 2e-5 * t.B * t.N, near


def test_tree_greedy_invalid_data():
    """Greedy trees on the flat stream's shape (64 trees of 5 nodes, V = 32000
    bf16): a malformed parent, a bad token at a tested child and a NaN in a
    reached row mark only their sequences; the others match the oracle."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_tree_inputs, bf16_bits
    t = make_tree_inputs(mode="greedy", B=64, N=5, V=32000, dtype="bf16", branching=(2,),
                         p_argmax=1.0, seed=12)
    assert sv.debug_flat_ctas(64, 4, 32000, "bf16") > 0
    t.par[1, 4] = 4                                    # malformed
    t.tok[2, 1] = 32000                                # first child of the root: tested
    t.logits[3, 0, 17] = bf16_bits(np.array([np.nan], np.float32))[0]  # the root row
    out, nodes, n, st, bits, _ = run_tree(t)
    ref = run_oracle(t)
    assert np.array_equal(n, ref.n) and np.array_equal(out, ref.out)
    assert np.array_equal(nodes, ref.nodes)
    assert list(n[1:4]) == [-1, -1, -1] and (n[4:] >= 0).all() and n[0] >= 0
    assert st == sv.SV_ERR_DATA
    want = sv.SV_DEV_BAD_TREE | sv.SV_DEV_BAD_TOKEN | sv.SV_DEV_BAD_ROW
    assert bits & want == want
