"""GPU parity of the n-gram (prompt-lookup) drafter against the oracle's rule.

"Decodificação especulativa explicada", §"A família de rascunhos" (prompt
lookup); "Speculative Decoding" (ch15), §"What proposes the tokens".  Drafts and
counts must equal the oracle's exactly (integer work).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_gpu_draft(hist, lengths, k, n_min, n_max):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    B = hist.shape[0]
    h = torch.from_numpy(np.ascontiguousarray(hist)).cuda()
    ln = torch.from_numpy(np.ascontiguousarray(lengths)).cuda()
    g = Guarded()
    d = g.empty((B, k), torch.int32, fill=-7)
    n = g.empty((B,), torch.int32, fill=-7)
    sv.spec_ngram_draft(h, ln, k, n_min, n_max, d, n)
    torch.cuda.synchronize()
    g.check()
    return d.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("k,n_min,n_max", [(4, 1, 4), (8, 2, 3), (5, 3, 32), (1, 1, 1)])
@pytest.mark.parametrize("Lmax,p_phrase", [(2000, 0.8), (300, 0.3), (5000, 0.95)])
def test_ngram_parity(k, n_min, n_max, Lmax, p_phrase):
    from speculative_decoding_verification_18_gb300.inputs import ngram_histories
    hist, lengths = ngram_histories(300, Lmax, V=32000, seed=Lmax + k, p_phrase=p_phrase)
    d, n = run_gpu_draft(hist, lengths, k, n_min, n_max)
    rd, rn = oracle.ngram_draft(hist, lengths, k, n_min, n_max)
    assert np.array_equal(n, rn) and np.array_equal(d, rd)
    assert (rn > 0).mean() > 0.3 if p_phrase > 0.5 else True


def test_ngram_edges():
    """Empty and one-token histories, lengths beyond Lmax or negative (clamped),
    runs of one token, a small vocabulary (many repeats)."""
    g = np.random.default_rng(1)
    hist = g.integers(0, 3, size=(12, 40)).astype(np.int32)
    hist[5] = 7
    lengths = np.array([0, 1, 2, 40, 55, 7, -3, 39, 3, 20, 33, 10], np.int32)
    for k, n_min, n_max in ((3, 1, 4), (6, 2, 32)):
        d, n = run_gpu_draft(hist, lengths, k, n_min, n_max)
        rd, rn = oracle.ngram_draft(hist, lengths, k, n_min, n_max)
        assert np.array_equal(n, rn) and np.array_equal(d, rd)


def test_ngram_large_history():
    from speculative_decoding_verification_18_gb300.inputs import ngram_histories
    hist, lengths = ngram_histories(8, 65536, V=50000, seed=3, p_phrase=0.9)
    d, n = run_gpu_draft(hist, lengths, 8, 1, 5)
    rd, rn = oracle.ngram_draft(hist, lengths, 8, 1, 5)
    assert np.array_equal(n, rn) and np.array_equal(d, rd)
