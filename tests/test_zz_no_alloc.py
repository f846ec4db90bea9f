"""The no-allocation sampled entry point against the workspace entry point.

Some callers cannot allocate device memory (operator plug-ins that only receive
their tensors, serving loops that forbid allocation after start-up), so
spec_verify_sample_noalloc keeps its scratch in a fixed array inside the
library.  This test calls it through the C ABI twice in a row, on two different
batches, and checks each result against spec_verify_sample with a caller-owned
workspace on the same inputs.  Outputs are integers, so the tolerance the other
tests use for integer outputs applies: exact equality.  It lives in its own file,
collected last, and passes alone in a fresh process as well as after the rest.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    assert torch.cuda.is_available()

    for seed, (B, k, V, dtype, T) in enumerate([(48, 5, 20011, "bf16", 0.8),
                                                 (33, 3, 4099, "f32", 1.1)]):
        inp = make_inputs(mode="sample", B=B, k=k, V=V, dtype=dtype, T=T, kind="zipf",
                          seed=500 + seed)
        if dtype == "bf16":
            lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).cuda()
        else:
            lg = torch.from_numpy(inp.logits).cuda()
        q = torch.from_numpy(inp.q).cuda()
        x = torch.from_numpy(inp.x).cuda()
        ua = torch.from_numpy(inp.ua).cuda()
        ur = torch.from_numpy(inp.ur).cuda()

        ref_out = torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda")
        ref_n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        ws = sv.workspace(B, k, V, lg.dtype)
        sv.spec_verify_sample(lg, q, x, ua, ur, T, ref_out, ref_n, ws)

        out = torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda")
        n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        sv.spec_verify_sample_noalloc(lg, q, x, ua, ur, T, out, n)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(n, ref_n)
        assert (n >= 0).all()


def test_noalloc_rejects_sizes_beyond_the_limit():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    from speculative_decoding_verification_18_gb300 import specverify as sv
    lib = sv.load()
    k = 7
    B = sv.SV_NOALLOC_MAX_ROWS // (k + 1) + 1
    P = 4096  # never dereferenced: the size check comes first
    st = lib.spec_verify_sample_noalloc(P, sv.SV_F32, P, P, P, P, 1.0, B, k, 100, P, P, None)
    assert st == sv.SV_ERR_WORKSPACE
