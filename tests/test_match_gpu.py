"""GPU parity of the sample-and-match verify (spec_verify_match) against the oracle.

"Decodificação especulativa explicada", §"A regra de amostragem por rejeição",
the simpler exact scheme: a target draw at every position, drafts kept while
they match.  Outputs must equal the oracle's MATCH mode token for token (a draw
may differ only when its uniform lies within ~1e-9 of a bin boundary: counted);
on the page's toy, acceptance must be sum_v p(v) q(v) and emitted tokens follow p.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import Guarded, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_match(inp, dev=None, tuning=None):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    dev = dev or to_device(inp)
    B, k, V = inp.B, inp.k, inp.V
    g = Guarded()
    out = g.empty((B, k + 1), torch.int32, fill=-7)
    n = g.empty((B,), torch.int32, fill=-7)
    ws = g.workspace(B, k, V, dev["logits"].dtype)
    sv.spec_verify_match(dev["logits"], dev["x"], dev["ua"], dev["ur"], inp.T, out, n, ws,
                         tuning=tuning)
    torch.cuda.synchronize()
    g.check()
    st, bits, _ = sv.spec_verify_read_status(ws)
    return out.cpu().numpy(), n.cpu().numpy(), st, bits


def _row_float64(inp, b, i):
    r = inp.logits[b, i]
    if inp.dtype == "bf16":
        return (r.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return r.astype(np.float64)


def compare_match(inp, out, n):
    """Hard mismatches and near-boundary ones (the first differing draw's uniform
    within 1e-9 of one of the oracle's bin edges on that row)."""
    ref = oracle.verify_batch(oracle.MATCH, inp.logits, inp.dtype, None, inp.x, inp.ua, inp.ur,
                              inp.T)
    hard, near = [], 0
    for b in np.nonzero((n != ref.n) | (out != ref.out).any(axis=1))[0]:
        if ref.n[b] < 0 or n[b] < 0:
            hard.append(int(b))
            continue
        j = int(np.nonzero(out[b] != ref.out[b])[0][0])
        u = float(inp.ua[b, j]) if j < inp.k else float(inp.ur[b])
        cdf = oracle.draw_cdf(_row_float64(inp, b, j), None, inp.T)
        if np.min(np.abs(np.concatenate([[0.0], cdf]) - u)) < 1e-9:
            near += 1
        else:
            hard.append(int(b))
    return ref, hard, near


SHAPES = [
    (1, 1, 1, "f32", 1.0), (3, 2, 2, "bf16", 0.7), (16, 4, 33, "bf16", 1.0),
    (64, 4, 100, "f32", 0.8), (40, 5, 4099, "bf16", 1.1), (9, 2, 40000, "bf16", 0.8),
    (7, 6, 65537, "f32", 1.0), (2, 3, 300001, "bf16", 1.0), (300, 3, 1000, "bf16", 0.9),
]


@pytest.mark.parametrize("B,k,V,dtype,T", SHAPES)
def test_match_small(B, k, V, dtype, T):
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    inp = make_inputs(mode="sample", B=B, k=k, V=V, dtype=dtype, T=T, kind="zipf",
                      draft_sigma=0.3, seed=B * 13 + V)
    out, n, st, bits = run_match(inp)
    ref, hard, near = compare_match(inp, out, n)
    assert not hard, hard[:5]
    assert near <= 1
    assert st == 0 and (bits & 0xF) == 0
    assert (n >= 0).all()


@pytest.mark.parametrize("name", ["c1", "c3", "c5"])
def test_match_workloads(name):
    from speculative_decoding_verification_18_gb300.inputs import workload
    inp = workload(name, seed=21)
    out, n, st, bits = run_match(inp)
    ref, hard, near = compare_match(inp, out, n)
    assert not hard, hard[:5]
    assert near <= 1


def test_match_precise_draws_only():
    """Every draw through the float-float pass."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    inp = make_inputs(mode="sample", B=24, k=4, V=70001, dtype="bf16", T=0.9, kind="zipf",
                      draft_sigma=0.3, seed=5)
    out, n, st, bits = run_match(inp, tuning=sv.Tuning(force_precise=1))
    ref, hard, near = compare_match(inp, out, n)
    assert not hard and near <= 1


def test_match_invalid_data():
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    inp = make_inputs(mode="sample", B=8, k=3, V=500, dtype="f32", T=1.0, kind="zipf",
                      draft_sigma=0.0, seed=9)
    inp.ua[1, 0] = 1.0            # bad uniform at position 0: always reached
    inp.ur[2] = -0.5              # bad bonus uniform: reached only if all k match
    inp.x[3, 0] = 10 ** 6         # bad draft token at position 0
    inp.logits[4, 0, 7] = np.nan  # bad row 0
    out, n, st, bits = run_match(inp)
    ref, hard, near = compare_match(inp, out, n)
    assert not hard
    assert n[1] == -1 and n[3] == -1 and n[4] == -1 and (out[[1, 3, 4]] == -1).all()
    assert (n[2] == -1) == (ref.n[2] == -1)
    assert st == 5 and (bits & 0xF) != 0  # SV_ERR_DATA with the error bits


def test_match_toy_acceptance_and_target_distribution():
    """One round with k = 1 from each context c of the page's toy: the draft
    survives with probability sum_v P[c, v] Q[c, v] and the emitted first token
    follows P[c] (200 000 sequences per context)."""
    from scipy.stats import chi2
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    P, Q = toy_language()
    N = 200_000
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    lnP = torch.from_numpy(np.log(P).astype(np.float32)).cuda()
    Qc = torch.cumsum(torch.from_numpy(Q.astype(np.float32)).cuda(), dim=1)
    for c in range(4):
        u = torch.rand(N, device="cuda", generator=g)
        x0 = torch.searchsorted(Qc[c].expand(N, 4).contiguous(),
                                (u * Qc[c, -1]).unsqueeze(1).contiguous(), right=True)
        x0 = x0.clamp_(max=3).to(torch.int32)
        logits = torch.stack([lnP[c].expand(N, 4), lnP[x0.squeeze(1).long()]], dim=1).contiguous()
        ud = torch.rand((N, 1), device="cuda", generator=g)
        ub = torch.rand(N, device="cuda", generator=g)
        gd = Guarded()
        out = gd.empty((N, 2), torch.int32)
        n = gd.empty(N, torch.int32)
        ws = gd.workspace(N, 1, 4, torch.float32)
        sv.spec_verify_match(logits, x0.contiguous(), ud, ub, 1.0, out, n, ws)
        torch.cuda.synchronize()
        gd.check()
        n = n.cpu().numpy()
        first = out[:, 0].cpu().numpy()
        beta = float((P[c] * Q[c]).sum())
        rate = (n >= 1).mean()
        assert abs(rate - beta) < 4 * np.sqrt(beta * (1 - beta) / N), (c, rate, beta)
        counts = np.bincount(first, minlength=4).astype(float)
        stat = float(((counts - N * P[c]) ** 2 / (N * P[c])).sum())
        assert chi2.sf(stat, 3) > 1e-4, (c, stat)
