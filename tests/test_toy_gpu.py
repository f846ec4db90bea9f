"""End-to-end generation through the C ABI, and the verify's fused bookkeeping.

The toy bigram language of "Decodificação especulativa explicada",
§"Amostragem especulativa em numpy, com prova", generated on the GPU with every
round verified by spec_verify_sample_kv: the sequences must follow the target's
exact joint (and must not follow the joint of the buggy "resample from p" rule,
computed by the oracle), and tokens per target pass must match the page's
measurement (§"Taxa de aceitação e tokens por passada").
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import exact as oexact
from conftest import read_golden
from parity import Guarded, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _chi2_pooled(counts, probs):
    """Pearson statistic and its upper-tail p-value, cells with < 5 expected hits
    pooled into one (the page's convention)."""
    from scipy.stats import chi2
    n = counts.sum()
    exp = n * probs
    big = exp >= 5
    obs_c = list(counts[big]) + ([counts[~big].sum()] if (~big).any() else [])
    exp_c = list(exp[big]) + ([exp[~big].sum()] if (~big).any() else [])
    obs_c, exp_c = np.array(obs_c, float), np.array(exp_c, float)
    stat = float(((obs_c - exp_c) ** 2 / exp_c).sum())
    return stat, float(chi2.sf(stat, len(obs_c) - 1))


def _dist_vector(dist, V, L):
    v = np.zeros(V ** L)
    for seq, p in dist.items():
        idx = 0
        for t in seq:
            idx = idx * V + t
        v[idx] = float(p)
    return v


@pytest.mark.parametrize("mode", ["sample", "greedy"])
@pytest.mark.parametrize("path", [1, 2, 3])
def test_kv_and_stats_epilogue(mode, path):
    """kv_len[b] += n + 1 for valid sequences only; the counters sum the round."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    inp = make_inputs(mode=mode, B=40, k=5, V=3001, dtype="bf16", T=0.9, kind="zipf",
                      p_argmax=0.6, seed=91)
    inp.x[3, 0] = inp.V + 5          # invalid draft token on a reached row
    if mode == "sample":
        inp.ur[7] = 1.5              # invalid uniform for the draw
    dev = to_device(inp)
    tu = sv.Tuning(path=path)
    ref_out, ref_n, _, _ = run_gpu(inp, dev, tuning=tu)
    B, k = inp.B, inp.k
    kv0 = torch.arange(100, 100 + B, dtype=torch.int32, device="cuda")
    gd = Guarded()
    kv = gd.empty(B, torch.int32)
    kv.copy_(kv0)
    stats = gd.empty(len(sv.STATS_FIELDS), torch.int64, fill=0)
    out = gd.empty((B, k + 1), torch.int32)
    n = gd.empty(B, torch.int32)
    ws = gd.workspace(B, k, inp.V, dev["logits"].dtype)
    if mode == "sample":
        sv.spec_verify_sample_kv(dev["logits"], dev["q"], dev["x"], dev["ua"], dev["ur"],
                                 inp.T, out, n, ws, kv_len=kv, stats=stats, tuning=tu)
    else:
        sv.spec_verify_greedy_kv(dev["logits"], dev["x"], out, n, ws, kv_len=kv, stats=stats,
                                 tuning=tu)
    torch.cuda.synchronize()
    gd.check()
    n = n.cpu().numpy()
    assert np.array_equal(n, ref_n) and np.array_equal(out.cpu().numpy(), ref_out)
    valid = n >= 0
    assert (~valid).sum() >= 1 and valid.sum() >= 30
    expect = kv0.cpu().numpy() + np.where(valid, n + 1, 0)
    assert np.array_equal(kv.cpu().numpy(), expect)
    st = sv.stats_dict(stats)
    nv = int(valid.sum())
    assert st == dict(rounds=nv, proposed=k * nv, accepted=int(n[valid].sum()),
                      emitted=int((n[valid] + 1).sum()), invalid=int((~valid).sum()))


def test_toy_generation_follows_the_exact_joint():
    """400 000 sequences of 4 tokens (k = 3), every round through the C ABI."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300 import toy
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    P, Q = toy_language()
    V, L, k, N = 4, 4, 3, 400_000
    models = toy.ToyModels.from_arrays(P, Q)
    seqs, length, stats = toy.generate(models, N, k, L, seed=2024)
    seqs = seqs.cpu().numpy().astype(np.int64)
    assert seqs.min() >= 0 and seqs.max() < V
    codes = ((seqs[:, 0] * V + seqs[:, 1]) * V + seqs[:, 2]) * V + seqs[:, 3]
    counts = np.bincount(codes, minlength=V ** L).astype(float)

    exact = _dist_vector(oexact.toy_exact_joint(P, L=L), V, L)
    buggy = _dist_vector(oexact.toy_sequence_distribution(
        P, Q, k=k, L=L, mode=oracle.SAMPLE_BUGGY), V, L)
    tv_exact = 0.5 * np.abs(counts / N - exact).sum()
    tv_buggy = 0.5 * np.abs(counts / N - buggy).sum()
    _, p_exact = _chi2_pooled(counts, exact)
    _, p_buggy = _chi2_pooled(counts, buggy)
    # The page's table at N = 400 000: speculative TV 0.0078, buggy 0.1075.
    assert tv_exact < 0.015, tv_exact
    assert p_exact > 1e-4, p_exact
    assert tv_buggy > 0.09 and p_buggy < 1e-12, (tv_buggy, p_buggy)

    st = sv.stats_dict(stats)
    length = length.cpu().numpy()
    assert length.min() >= L and length.max() <= L + k
    assert st["invalid"] == 0
    assert st["emitted"] == int(length.sum())
    assert st["accepted"] == st["emitted"] - st["rounds"]
    assert st["proposed"] == k * st["rounds"]


def test_toy_tokens_per_target_pass_match_the_page():
    """2048 chains x 100 rounds per k, against the page's 50 000-round table: the
    page's figures carry a standard error near 0.004 (tokens) and 0.002 (alpha);
    ours about half that."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300 import toy
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    P, Q = toy_language()
    models = toy.ToyModels.from_arrays(P, Q)
    for row in read_golden("tokens_per_call.txt"):
        k, alpha_page, tpc_page = int(row[0]), float(row[1]), float(row[2])
        stats, judged = toy.chains(models, B=2048, steps=100, k=k, seed=7 + k)
        st = sv.stats_dict(stats)
        tpc = st["emitted"] / st["rounds"]
        alpha = st["accepted"] / judged
        assert st["rounds"] == 2048 * 100 and st["invalid"] == 0
        assert abs(tpc - tpc_page) < 0.03, (k, tpc, tpc_page)
        assert abs(alpha - alpha_page) < 0.012, (k, alpha, alpha_page)
