"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA path
through the C ABI, run the oracle, and compare with near-threshold accounting.

Parity rule (floating point decides an integer here, so exact equality is not
always attainable): greedy outputs must be bit-exact; in sampled mode every
integer output must be equal, except that a sequence whose first differing
decision had its uniform within 1e-5 of the oracle's threshold (min(1, p/q) for
an accept test, a bin boundary C_{t-1}/C_tot or C_t/C_tot for a draw) is counted
as a near-threshold mismatch; those must stay below 1e-5 of all rows.
Row statistics must agree to 1e-5 relative.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_U = 1e-5
TOL_STATS = 1e-5

GUARD_BYTES = 256      # guard bytes on each side of a device buffer (keeps 256-byte alignment)
GUARD_PATTERN = 0xA5


class Guarded:
    """Device buffers that the library writes, each with GUARD_BYTES of a known
    pattern on both sides.  ``check()`` fails if a call wrote past either end of
    any of them: a host-side stand-in for a memory checker, since writes out of
    bounds are otherwise invisible to tests that read only the intended
    elements.  Nothing here touches memory the buffers do not own."""

    def __init__(self, device="cuda"):
        self.device = device
        self.bufs = []

    def empty(self, shape, dtype, fill=None):
        shape = tuple(int(d) for d in (shape if isinstance(shape, (tuple, list)) else (shape,)))
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), GUARD_PATTERN,
                         dtype=torch.uint8, device=self.device)
        view = raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
        if fill is not None:
            view.fill_(fill)
        self.bufs.append((raw, nbytes))
        return view

    def workspace(self, B, k, V, dtype=torch.bfloat16):
        from speculative_decoding_verification_18_gb300 import specverify as sv
        n = sv.spec_verify_workspace_size(B, k, V, sv.SV_BF16 if dtype == torch.bfloat16
                                          else sv.SV_F32)
        return self.empty((max(n, 256),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, nbytes) in enumerate(self.bufs):
            head = raw[:GUARD_BYTES]
            tail = raw[GUARD_BYTES + nbytes:]
            ok_h = bool((head == GUARD_PATTERN).all())
            ok_t = bool((tail == GUARD_PATTERN).all())
            assert ok_h and ok_t, f"guard bytes of buffer {i} ({nbytes} bytes) overwritten " \
                                  f"({'before' if not ok_h else ''}{' after' if not ok_t else ''})"


def to_device(inp, device="cuda"):
    """Device copies of one VerifyInputs batch."""
    if inp.dtype == "bf16":
        lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16)
    else:
        lg = torch.from_numpy(inp.logits)
    d = dict(logits=lg.to(device), x=torch.from_numpy(inp.x).to(device))
    if inp.mode == "sample":
        d["q"] = torch.from_numpy(inp.q).to(device)
        d["ua"] = torch.from_numpy(inp.ua).to(device)
        d["ur"] = torch.from_numpy(inp.ur).to(device)
    return d


def run_gpu(inp, dev=None, ws=None, two_stage=False, tuning=None):
    """One verify of `inp` through the C ABI (with the per-call options `tuning`,
    an sv.Tuning, or the automatic choices).  The outputs (and the workspace,
    unless one is given) carry guard bytes, checked after the call."""
    from speculative_decoding_verification_18_gb300 import specverify as sv
    dev = dev or to_device(inp)
    B, k, V = inp.B, inp.k, inp.V
    g = Guarded()
    out = g.empty((B, k + 1), torch.int32, fill=-7)
    n = g.empty((B,), torch.int32, fill=-7)
    if ws is None:
        ws = g.workspace(B, k, V, dev["logits"].dtype)
    if inp.mode == "greedy":
        if two_stage:
            sv.spec_verify_rows(sv.SV_MODE_GREEDY, dev["logits"], None, dev["x"], 1.0, ws,
                                tuning=tuning)
            sv.spec_verify_finish(sv.SV_MODE_GREEDY, dev["logits"], None, dev["x"], None, None,
                                  1.0, out, n, ws, tuning=tuning)
        else:
            sv.spec_verify_greedy(dev["logits"], dev["x"], out, n, ws, tuning=tuning)
    else:
        if two_stage:
            sv.spec_verify_rows(sv.SV_MODE_SAMPLE, dev["logits"], dev["q"], dev["x"], inp.T, ws,
                                tuning=tuning)
            sv.spec_verify_finish(sv.SV_MODE_SAMPLE, dev["logits"], dev["q"], dev["x"], dev["ua"],
                                  dev["ur"], inp.T, out, n, ws, tuning=tuning)
        else:
            sv.spec_verify_sample(dev["logits"], dev["q"], dev["x"], dev["ua"], dev["ur"], inp.T,
                                  out, n, ws, tuning=tuning)
    torch.cuda.synchronize()
    g.check()
    st, bits, ndeg = sv.spec_verify_read_status(ws)
    stats = sv.spec_verify_row_stats(ws, B, k)
    return out.cpu().numpy(), n.cpu().numpy(), stats, (st, bits, ndeg)


def run_oracle(inp):
    mode = oracle.GREEDY if inp.mode == "greedy" else oracle.SAMPLE
    return oracle.verify_batch(mode, inp.logits, inp.dtype, inp.q, inp.x, inp.ua, inp.ur,
                               inp.T if inp.mode == "sample" else 1.0)


Report = oracle.Comparison


def compare_outputs(inp, out, n, ref) -> Report:
    """The CUDA path's integer outputs against the oracle's (parity rule above)."""
    return oracle.compare_outputs(inp.mode, inp.ua, inp.ur, out, n, ref, TOL_U)


def compare_stats(inp, stats, ref, n=None, check_sum=True):
    """Row statistics of every row the GPU scan read (rows it never reached carry
    NaN): argmax and max exact, S to 1e-5 relative, q(x) exact, and p(x) to 1e-5
    relative on the rows the scan judged (0..n in sampled mode)."""
    T = inp.T if inp.mode == "sample" else 1.0
    read = np.isfinite(stats["m"])
    assert read[:, 0].all(), "row 0 must always be read"
    if n is not None:  # every row up to the decision row was read
        for b in range(inp.B):
            if n[b] >= 0:
                assert read[b, :n[b] + 1].all()
    assert np.array_equal(stats["argmax"][read], ref.row_argmax[read]), "argmax differs"
    # the oracle reports max_j l_j / T in double; the GPU keeps the raw max
    m_gpu = stats["m"].astype(np.float64) / np.float64(np.float32(T))
    fin = read & np.isfinite(ref.row_m)
    assert np.array_equal(m_gpu[fin], ref.row_m[fin]), "row max differs"
    if inp.mode == "sample" and check_sum:
        ok = read & np.isfinite(ref.row_S)
        rel = np.abs(stats["S"][ok] - ref.row_S[ok]) / ref.row_S[ok]
        assert rel.size == 0 or rel.max() < TOL_STATS, f"S rel err {rel.max():.3g}"
        judged = np.zeros_like(read)
        if n is not None:
            for b in range(inp.B):
                judged[b, :min(int(n[b]), inp.k - 1) + 1] = n[b] >= 0
        px_ref = ref.row_px
        px = stats["px"].astype(np.float64)
        ok = judged & np.isfinite(px_ref) & (px_ref > 1e-37)
        ok[:, inp.k] = False
        rel = np.abs(px[ok] - px_ref[ok]) / px_ref[ok]
        assert rel.size == 0 or rel.max() < TOL_STATS, f"p(x) rel err {rel.max():.3g}"
        qx_ref = ref.row_qx[:, :inp.k]
        ok = read[:, :inp.k] & np.isfinite(qx_ref)
        assert np.array_equal(stats["qx"][:, :inp.k][ok].astype(np.float64), qx_ref[ok])
