"""Parity at scale: the large workloads' shapes over at least 10^6 seeded rows
each, and config-1-shaped inputs over 10^6 sequences.

The parity rule allows a sampled output to differ from the oracle's only where
the first differing decision had its uniform within 1e-5 of the oracle's
threshold, and such near-threshold cases must stay below 1 in 10^5 rows
("Decodificação especulativa explicada", §"A regra de amostragem por rejeição":
the rule is exact, so any other difference is an error).  A rate needs many
rows: each test generates one set of logits and q with the workload's sizes,
dtype, temperature and value distributions (more sequences than the workload
has, so that the oracle's threads stay busy), then verifies it again and again
with freshly drawn drafts (from q) and fresh uniforms, in launches of the
workload's own batch size so that the GPU takes the workload's own path.  The
oracle gets the row statistics it computed once for these logits
(verify_batch_stats), which is what lets it keep up.

Config 1 (V = 32, k = 4): one instance tiled over 10^6 sequences with fresh
drafts and uniforms, every output compared with the oracle's, then the emitted
token at each position tested against p (chi-square) and the mean accepted
length against the product of the per-position acceptance rates.
"""
import math
import os
import time

import numpy as np
import pytest
import torch

import oracle
from parity import TOL_U, Guarded

pytestmark = pytest.mark.gpu

ROWS = int(os.environ.get("SV_PARITY_SWEEP_ROWS", "1000000"))
RATE = 1e-5

# workload: (sequences generated, sequences per launch = the workload's B)
SWEEPS = {"c3": (128, 32), "c4": (256, 256), "c5": (64, 1)}


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _aligned(t):
    """The ABI takes 16-byte aligned pointers: a slice that is not gets a copy."""
    return t if t.data_ptr() % 16 == 0 else t.clone()


def _device_logits(inp):
    if inp.dtype == "bf16":
        return torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(inp.logits).cuda()


@pytest.mark.parametrize("name", sorted(SWEEPS))
def test_mismatch_rate_over_a_million_rows(name):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import WORKLOADS, make_inputs, redraw
    params = dict(WORKLOADS[name])
    B_big, B_launch = SWEEPS[name]
    assert B_launch == params["B"]
    params.update(B=B_big, seed=9000 + int(name[1]))
    t0 = time.perf_counter()
    inp = make_inputs(**params)
    k, V, T = inp.k, inp.V, inp.T
    per_rep = B_big * (k + 1)
    reps = -(-ROWS // per_rep)
    rd = redraw(inp, reps, seed=9100 + int(name[1]))
    stats = oracle.row_stats_batch(inp.logits, inp.dtype, T)
    assert not stats.bad.any()
    lg = _device_logits(inp)
    q = torch.from_numpy(inp.q).cuda()
    path = sv.debug_path(sv.SV_MODE_SAMPLE, B_launch, V, inp.dtype)
    nl = B_big // B_launch
    g = Guarded()
    outs = [g.empty((B_launch, k + 1), torch.int32) for _ in range(nl)]
    ns = [g.empty(B_launch, torch.int32) for _ in range(nl)]
    wss = [g.workspace(B_launch, k, V, lg.dtype) for _ in range(nl)]
    t_setup = time.perf_counter() - t0
    near = hard = differing = 0
    precise = counted = 0  # draws that needed the float-float pass, over the first reps
    for r in range(reps):
        x = torch.from_numpy(rd.x[r]).cuda()
        ua = torch.from_numpy(rd.ua[r]).cuda()
        ur = torch.from_numpy(rd.ur[r]).cuda()
        for j in range(nl):
            b0, b1 = j * B_launch, (j + 1) * B_launch
            sv.spec_verify_sample(lg[b0:b1], q[b0:b1], _aligned(x[b0:b1]), _aligned(ua[b0:b1]),
                                  _aligned(ur[b0:b1]), T, outs[j], ns[j], wss[j])
        if r < 200:
            for j in range(nl):
                precise += sv.debug_status_counts(wss[j])[5]
            counted += B_big
        ref = oracle.verify_batch_stats(oracle.SAMPLE, inp.logits, inp.dtype, inp.q, rd.x[r],
                                        rd.ua[r], rd.ur[r], T, stats)
        out = torch.cat(outs).cpu().numpy()
        n = torch.cat(ns).cpu().numpy()
        c = oracle.compare_outputs("sample", rd.ua[r], rd.ur[r], out, n, ref, TOL_U)
        assert c.hard == 0, (name, r, c.hard_detail)
        near += c.near_threshold
        hard += c.hard
        differing += c.mismatched_sequences
        assert (ref.n >= 0).all()
    g.check()
    rows = reps * per_rep
    print(f"\n{name} (path {path}): {rows} rows in {reps} x {nl} launches of B={B_launch}, "
          f"{differing} differing sequences, {near} near-threshold "
          f"(rate {near / rows:.2e}, limit {RATE:.0e}), {hard} hard; precise draws "
          f"{precise}/{counted} ({precise / max(counted, 1):.2%}); "
          f"setup {t_setup:.1f} s, total {time.perf_counter() - t0:.1f} s")
    assert rows >= ROWS
    assert hard == 0
    assert near <= RATE * rows


def _softmax64(l, T):
    z = np.asarray(l, dtype=np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def test_config1_shape_million_sequences():
    """Config 1 over 10^6 sequences: element-by-element parity, then the
    statistics of the GPU's outputs against what the pages fix (the emitted token
    at position i follows p_i given that position i is reached, [DEE]
    §"Amostragem especulativa em numpy, com prova"; the chance of reaching
    position i is the product of the acceptance rates alpha_j = sum min(p_j, q_j),
    [DEE] §"Taxa de aceitação e tokens por passada")."""
    from scipy.stats import chi2

    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import (WORKLOADS, VerifyInputs,
                                                                   make_inputs, redraw)
    one = make_inputs(**WORKLOADS["c1"])
    B = max(ROWS, 1)
    k, V, T = one.k, one.V, one.T
    rd = redraw(one, B, seed=9201)
    x = rd.x.reshape(B, k)
    ua = rd.ua.reshape(B, k)
    ur = rd.ur.reshape(B)
    logits = np.ascontiguousarray(np.broadcast_to(one.logits, (B, k + 1, V)))
    qq = np.ascontiguousarray(np.broadcast_to(one.q, (B, k, V)))
    inp = VerifyInputs("sample", "f32", B, k, V, T, logits, qq, x, ua, ur)

    g = Guarded()
    out_d = g.empty((B, k + 1), torch.int32, fill=-7)
    n_d = g.empty(B, torch.int32, fill=-7)
    ws = g.workspace(B, k, V, torch.float32)
    sv.spec_verify_sample(torch.from_numpy(logits).cuda(), torch.from_numpy(qq).cuda(),
                          torch.from_numpy(x).cuda(), torch.from_numpy(ua).cuda(),
                          torch.from_numpy(ur).cuda(), T, out_d, n_d, ws)
    torch.cuda.synchronize()
    g.check()
    out, n = out_d.cpu().numpy(), n_d.cpu().numpy()

    st1 = oracle.row_stats_batch(one.logits, "f32", T)
    tile = lambda a: np.ascontiguousarray(np.broadcast_to(a, (B, k + 1)))
    stats = oracle.RowStats(tile(st1.m), tile(st1.S), tile(st1.argmax), tile(st1.bad))
    ref = oracle.verify_batch_stats(oracle.SAMPLE, logits, "f32", qq, x, ua, ur, T, stats)
    c = oracle.compare_outputs("sample", ua, ur, out, n, ref, TOL_U)
    print(f"\nconfig 1 x {B}: {c.mismatched_sequences} differing sequences, "
          f"{c.near_threshold} near-threshold, {c.hard} hard")
    assert c.hard == 0, c.hard_detail
    assert c.near_threshold <= RATE * B * (k + 1)

    lvals = one.logits[0].astype(np.float64)
    p = np.stack([_softmax64(lvals[i], T) for i in range(k + 1)])
    qd = one.q[0].astype(np.float64)
    alpha = np.minimum(p[:k], qd).sum(axis=1)
    for i in range(k + 1):
        reached = n >= i
        m = int(reached.sum())
        counts = np.bincount(out[reached, i], minlength=V).astype(float)
        expect = m * p[i]
        order = np.argsort(expect)  # pool the smallest cells until each has >= 5
        obs_c, exp_c, acc_o, acc_e = [], [], 0.0, 0.0
        for j in order:
            acc_o += counts[j]
            acc_e += expect[j]
            if acc_e >= 5.0:
                obs_c.append(acc_o)
                exp_c.append(acc_e)
                acc_o = acc_e = 0.0
        if acc_e > 0 and exp_c:
            obs_c[-1] += acc_o
            exp_c[-1] += acc_e
        obs_c, exp_c = np.array(obs_c), np.array(exp_c)
        stat = float(((obs_c - exp_c) ** 2 / exp_c).sum())
        pval = chi2.sf(stat, len(exp_c) - 1)
        print(f"position {i}: {m} sequences reach it, chi2 {stat:.1f} on {len(exp_c) - 1} dof, "
              f"p {pval:.3f}")
        assert pval > 1e-4, (i, stat, pval)
    # E[n] = sum_{i=1..k} prod_{j<i} alpha_j
    en = sum(math.prod(alpha[:i]) for i in range(1, k + 1))
    se = n.std() / math.sqrt(B)
    print(f"mean accepted {n.mean():.5f}, expected {en:.5f} (4 SE = {4 * se:.5f})")
    assert abs(n.mean() - en) < 4 * se
