"""Host-side pieces of the toy generation driver (no GPU)."""
import numpy as np
import torch

from oracle import exact as oexact


def test_toy_language_is_the_oracles():
    """The input module's bigram toy is the oracle's: both follow the page's
    generator calls ("Decodificação especulativa explicada", §"Amostragem
    especulativa em numpy, com prova")."""
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    P, Q = toy_language()
    P2, Q2 = oexact.toy_bigram()
    assert np.array_equal(P, P2) and np.array_equal(Q, Q2)
    # the page's printed acceptance per context
    assert np.allclose(np.minimum(P, Q).sum(axis=1), [0.672, 0.692, 0.856, 0.863], atol=5e-4)


def test_toy_models_tables():
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    from speculative_decoding_verification_18_gb300.toy import ToyModels
    P, Q = toy_language()
    m = ToyModels.from_arrays(P, Q, device="cpu")
    assert m.V == 4 and m.lnP.shape == (4, 4) and m.Q.dtype == torch.float32
    assert torch.allclose(torch.softmax(m.lnP, dim=1), torch.from_numpy(P).float(), atol=1e-6)
    assert torch.allclose(m.Qc[:, -1], torch.ones(4), atol=1e-6)


def test_toy_exact_joint_is_the_oracles():
    """The driver's report compares against the target's joint; it must be the
    oracle's plain target-only joint, sequence for sequence."""
    from speculative_decoding_verification_18_gb300.inputs import toy_language
    from speculative_decoding_verification_18_gb300.toy import exact_joint
    P, _ = toy_language()
    for L in (1, 2, 4):
        J = exact_joint(P, L)
        for seq, p in oexact.toy_exact_joint(P, L=L).items():
            idx = 0
            for t in seq:
                idx = idx * 4 + t
            assert abs(J[idx] - float(p)) < 1e-15
