"""The no-allocation sampled entry point against the workspace entry point.

Some callers cannot allocate device memory (operator plug-ins that only receive
their tensors, serving loops that forbid allocation after start-up), so
spec_verify_sample_noalloc keeps its scratch in a fixed array inside the
library.  These tests call it through the C ABI, several times in a row on
different batches (the paths that keep only row records there, the
row-skipping path whose stop rows and deferred precise-draw list also live
there, and a batch of exactly the largest accepted row count), and check each
result against spec_verify_sample with a caller-owned workspace on the same
inputs; every output buffer carries guard bytes.  Outputs are integers, so the
tolerance the other tests use for integer outputs applies: exact equality.  The
file is collected last, and passes alone in a fresh process as well as after the
rest.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _run_pair(sv, inp):
    """spec_verify_sample with a caller workspace, then the no-allocation entry
    point on the same inputs; both sets of outputs carry guard bytes."""
    from parity import Guarded
    B, k, V, T = inp.B, inp.k, inp.V, inp.T
    if inp.dtype == "bf16":
        lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        lg = torch.from_numpy(inp.logits).cuda()
    q = torch.from_numpy(inp.q).cuda()
    x = torch.from_numpy(inp.x).cuda()
    ua = torch.from_numpy(inp.ua).cuda()
    ur = torch.from_numpy(inp.ur).cuda()
    g = Guarded()
    ref_out = g.empty((B, k + 1), torch.int32, fill=-7)
    ref_n = g.empty((B,), torch.int32, fill=-7)
    ws = g.workspace(B, k, V, lg.dtype)
    sv.spec_verify_sample(lg, q, x, ua, ur, T, ref_out, ref_n, ws)
    _, bits, _ = sv.spec_verify_read_status(ws)
    out = g.empty((B, k + 1), torch.int32, fill=-7)
    n = g.empty((B,), torch.int32, fill=-7)
    sv.spec_verify_sample_noalloc(lg, q, x, ua, ur, T, out, n)
    torch.cuda.synchronize()
    g.check()
    assert torch.equal(out, ref_out) and torch.equal(n, ref_n)
    assert (n >= 0).all()
    return bits


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
        _run_pair(sv, inp)


def test_noalloc_row_skipping_path_and_precise_list():
    """A batch large enough for the row-skipping path: its stop rows and its list
    of deferred precise draws live in the library's array too.  A long-tailed
    fp32 vocabulary makes some draws need the precise pass, so the list is used
    (the workspace run reports it)."""
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    B, k = 96, 4
    assert sv.debug_path(sv.SV_MODE_SAMPLE, B, 151936, "f32") == sv.PATH_SKIP
    inp = make_inputs(mode="sample", B=B, k=k, V=151936, dtype="f32", T=1.0, kind="zipf",
                      slope=1.0, noise=1.5, draft_sigma=1.0, seed=610)
    bits = _run_pair(sv, inp)
    assert bits & sv.SV_DEV_PRECISE


def test_noalloc_at_the_row_limit():
    """Exactly SV_NOALLOC_MAX_ROWS rows (B = 3000, k = 8) on the row-skipping path."""
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    from speculative_decoding_verification_18_gb300 import specverify as sv
    from speculative_decoding_verification_18_gb300.inputs import make_inputs
    B, k = sv.SV_NOALLOC_MAX_ROWS // 9, 8
    assert B * (k + 1) == sv.SV_NOALLOC_MAX_ROWS
    assert sv.debug_path(sv.SV_MODE_SAMPLE, B, 64, "f32") == sv.PATH_SKIP
    inp = make_inputs(mode="sample", B=B, k=k, V=64, dtype="f32", T=1.0, kind="gauss",
                      scale=2.0, draft_sigma=0.5, seed=611)
    _run_pair(sv, inp)


def test_noalloc_rejects_sizes_beyond_the_limit():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    from speculative_decoding_verification_18_gb300 import specverify as sv
    lib = sv.load()
    P = 4096  # never dereferenced: the size check comes first
    for k in (7, 8):
        B = sv.SV_NOALLOC_MAX_ROWS // (k + 1) + 1
        st = lib.spec_verify_sample_noalloc(P, sv.SV_F32, P, P, P, P, 1.0, B, k, 100, P, P,
                                            None)
        assert st == sv.SV_ERR_WORKSPACE
