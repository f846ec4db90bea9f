"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments synchronously, before touching the CUDA runtime."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADERS = [os.path.join(ROOT, "include", h) for h in ("specverify.h", "specverify_debug.h")]


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_18_gb300 import build
    build.build()
    from speculative_decoding_verification_18_gb300 import specverify
    return specverify.load()


def declared():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(spec_verify_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size(lib):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    # header, 5 row records per sequence, status and stop words, the precise
    # list (a 16-byte counter and B entries); then the split draw's region:
    # five words per sequence (arrival counters, the precise entry's ambiguous
    # count, normaliser and margin), 32 ambiguous-element slots of 16 bytes,
    # 5 slice sums of 32 bytes (V = 32000: 4000 chunks of 8, 5 slices), 512
    # precise item sums of 32 bytes, and 16 bytes of block sums per 64 elements
    # of each decision row; then per row an arrival counter, 8 partials of 16
    # bytes and a 16-byte gather record (the split row-skipping stream);
    # rounded to 256
    base = 256 + 64 * 5 * 32 + 64 * 4 * 2 + 16 + 64 * 4
    split = 64 * 5 * 4 + 64 * 32 * 16 + 64 * 5 * 32 + 512 * 32 + 64 * 500 * 16
    rows = 320 * 4 + 320 * 8 * 16 + 320 * 16
    assert sv.spec_verify_workspace_size(64, 4, 32000) == -(-(base + split + rows) // 256) * 256
    # one sequence: 368 bytes before the split region, which holds 512 precise
    # item sums of 32 bytes whatever the batch
    assert sv.spec_verify_workspace_size(1, 1, 1) == 17664
    assert sv.spec_verify_workspace_size(0, 4, 10) == 512
    assert sv.spec_verify_workspace_size(1, 0, 10) == 0
    assert sv.spec_verify_workspace_size(1, 65, 10) == 0
    assert sv.spec_verify_workspace_size(1, 4, (1 << 21) + 1) == 0
    assert sv.spec_verify_workspace_size(1, 4, 10, 7) == 0


def test_argument_errors_without_gpu(lib):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    P = 4096  # a 16-byte-aligned fake address: never dereferenced on these paths
    ws = sv.spec_verify_workspace_size(2, 3, 100)
    args = lambda **kw: dict(dict(l=P, dt=sv.SV_F32, q=P, x=P, ua=P, ur=P, T=1.0, B=2, k=3,
                                  V=100, out=P, n=P, ws=P, wsb=ws), **kw)

    def sample(**kw):
        a = args(**kw)
        return lib.spec_verify_sample(a["l"], a["dt"], a["q"], a["x"], a["ua"], a["ur"], a["T"],
                                      a["B"], a["k"], a["V"], a["out"], a["n"], a["ws"], a["wsb"],
                                      None)

    assert sample(l=None) == sv.SV_ERR_INVALID_ARG
    assert sample(q=None) == sv.SV_ERR_INVALID_ARG
    assert sample(T=0.0) == sv.SV_ERR_INVALID_ARG
    assert sample(T=float("nan")) == sv.SV_ERR_INVALID_ARG
    assert sample(T=float("inf")) == sv.SV_ERR_INVALID_ARG
    assert sample(l=P + 2) == sv.SV_ERR_INVALID_ARG           # misaligned
    assert sample(ws=None) == sv.SV_ERR_WORKSPACE
    assert sample(wsb=ws - 1) == sv.SV_ERR_WORKSPACE
    assert sample(k=65, wsb=1 << 20) == sv.SV_ERR_UNSUPPORTED
    assert sample(V=0) == sv.SV_ERR_INVALID_ARG
    assert sample(B=-1) == sv.SV_ERR_INVALID_ARG
    assert sample(dt=9) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_greedy(None, 0, P, 2, 3, 100, P, P, P, ws, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_greedy(P, 0, P, 2, 3, 100, None, P, P, ws, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_rows(7, P, 0, P, P, 1.0, 2, 3, 100, P, ws, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_read_status(None, None, None, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_debug_ffexp(None, 0.0, 1.0, 5, None, None) == sv.SV_ERR_INVALID_ARG


def test_status_strings(lib):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    seen = {sv.status_string(s) for s in range(7)}
    assert len(seen) == 7 and "ok" in seen
    assert sv.status_string(99) == "unknown status"


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    monkeypatch.setattr(sv, "_lib", None)
    monkeypatch.setattr(sv, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        sv.load()


def test_ngram_argument_errors(lib):
    """Argument errors come back before any launch (no GPU needed)."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    f = lib.spec_ngram_draft
    assert f(None, None, 1, 10, 4, 1, 4, None, None, None) == sv.SV_ERR_INVALID_ARG
    assert f(None, None, 0, 10, 0, 1, 4, None, None, None) == sv.SV_ERR_INVALID_ARG   # k < 1
    assert f(None, None, 0, 10, 65, 1, 4, None, None, None) == sv.SV_ERR_INVALID_ARG  # k > 64
    assert f(None, None, 0, 10, 4, 0, 4, None, None, None) == sv.SV_ERR_INVALID_ARG  # n_min < 1
    assert f(None, None, 0, 10, 4, 3, 2, None, None, None) == sv.SV_ERR_INVALID_ARG  # n_max < n_min
    assert f(None, None, 0, 10, 4, 1, 33, None, None, None) == sv.SV_ERR_INVALID_ARG  # n_max > 32
    assert f(None, None, -1, 10, 4, 1, 4, None, None, None) == sv.SV_ERR_INVALID_ARG  # B < 0


def test_tree_argument_errors(lib):
    """spec_verify_tree rejects bad arguments before any launch (no GPU needed)."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    P = 4096
    ws = sv.spec_verify_workspace_size(2, 4, 100)

    def tree(mode=sv.SV_MODE_SAMPLE, l=P, q=P, tok=P, par=P, ua=P, ur=P, T=1.0, B=2, N=5,
             V=100, out=P, nodes=P, n=P, wsp=P, wsb=ws):
        return lib.spec_verify_tree(mode, l, sv.SV_F32, q, tok, par, ua, ur, T, B, N, V, out,
                                    nodes, n, wsp, wsb, None)

    assert tree(mode=7) == sv.SV_ERR_INVALID_ARG
    assert tree(N=1) == sv.SV_ERR_INVALID_ARG
    assert tree(N=66, wsb=1 << 20) == sv.SV_ERR_UNSUPPORTED
    assert tree(par=None) == sv.SV_ERR_INVALID_ARG
    assert tree(nodes=None) == sv.SV_ERR_INVALID_ARG
    assert tree(tok=P + 4) == sv.SV_ERR_INVALID_ARG
    assert tree(q=None) == sv.SV_ERR_INVALID_ARG
    assert tree(T=0.0) == sv.SV_ERR_INVALID_ARG
    assert tree(wsb=ws - 1) == sv.SV_ERR_WORKSPACE
    # greedy needs no q, uniforms or temperature: its errors are the others
    assert tree(mode=sv.SV_MODE_GREEDY, q=None, ua=None, ur=None, T=0.0,
                par=None) == sv.SV_ERR_INVALID_ARG


def test_tuning_options_are_per_call_and_checked(lib):
    """The test and tuning options travel with the call (sv_tuning): there is no
    process-wide setter left in the library, and an out-of-range option is an
    argument error returned before any launch."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    for gone in ("spec_verify_debug_force_path", "spec_verify_debug_force_precise",
                 "spec_verify_debug_draw_split", "spec_verify_debug_precise_split",
                 "spec_verify_debug_rows_split", "spec_verify_debug_flat",
                 "spec_verify_debug_fused_tuning"):
        assert not hasattr(lib, gone), gone
    P = 4096
    ws = sv.spec_verify_workspace_size(2, 3, 100)
    for bad in (dict(path=4), dict(path=-1), dict(draw_split=3), dict(precise_split=32),
                dict(rows_split=5), dict(rows_threads=200), dict(fused_defer=3),
                dict(fused_pad_kib=161), dict(draw_mode=3)):
        t = sv.Tuning(**bad)
        st = lib.spec_verify_sample_tuned(P, sv.SV_F32, P, P, P, P, 1.0, 2, 3, 100, P, P, P, ws,
                                          None, None, None, ctypes.byref(t))
        assert st == sv.SV_ERR_INVALID_ARG, bad
        st = lib.spec_verify_greedy_tuned(P, sv.SV_F32, P, 2, 3, 100, P, P, P, ws, None, None,
                                          None, ctypes.byref(t))
        assert st == sv.SV_ERR_INVALID_ARG, bad
