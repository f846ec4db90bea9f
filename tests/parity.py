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

from dataclasses import dataclass

import numpy as np
import torch

import oracle

TOL_U = 1e-5
TOL_STATS = 1e-5


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


def run_gpu(inp, dev=None, ws=None, two_stage=False):
    from speculative_decoding_verification_18_gb300 import specverify as sv
    dev = dev or to_device(inp)
    B, k, V = inp.B, inp.k, inp.V
    out = torch.full((B, k + 1), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = sv.workspace(B, k, V, dev["logits"].dtype)
    if inp.mode == "greedy":
        if two_stage:
            sv.spec_verify_rows(sv.SV_MODE_GREEDY, dev["logits"], None, dev["x"], 1.0, ws)
            sv.spec_verify_finish(sv.SV_MODE_GREEDY, dev["logits"], None, dev["x"], None, None,
                                  1.0, out, n, ws)
        else:
            sv.spec_verify_greedy(dev["logits"], dev["x"], out, n, ws)
    else:
        if two_stage:
            sv.spec_verify_rows(sv.SV_MODE_SAMPLE, dev["logits"], dev["q"], dev["x"], inp.T, ws)
            sv.spec_verify_finish(sv.SV_MODE_SAMPLE, dev["logits"], dev["q"], dev["x"], dev["ua"],
                                  dev["ur"], inp.T, out, n, ws)
        else:
            sv.spec_verify_sample(dev["logits"], dev["q"], dev["x"], dev["ua"], dev["ur"], inp.T,
                                  out, n, ws)
    torch.cuda.synchronize()
    st, bits, ndeg = sv.spec_verify_read_status(ws)
    stats = sv.spec_verify_row_stats(ws, B, k)
    return out.cpu().numpy(), n.cpu().numpy(), stats, (st, bits, ndeg)


def run_oracle(inp):
    mode = oracle.GREEDY if inp.mode == "greedy" else oracle.SAMPLE
    return oracle.verify_batch(mode, inp.logits, inp.dtype, inp.q, inp.x, inp.ua, inp.ur,
                               inp.T if inp.mode == "sample" else 1.0)


@dataclass
class Report:
    rows: int
    sequences: int
    mismatched_sequences: int
    near_threshold: int
    hard: int
    hard_detail: list


def compare_outputs(inp, out, n, ref) -> Report:
    B, k = inp.B, inp.k
    near = hard = mism = 0
    detail = []
    for b in range(B):
        if n[b] == ref.n[b] and np.array_equal(out[b], ref.out[b]):
            continue
        mism += 1
        if inp.mode == "greedy" or n[b] < 0 or ref.n[b] < 0:
            hard += 1
            detail.append((b, "greedy/invalid", int(n[b]), int(ref.n[b])))
            continue
        if n[b] != ref.n[b]:
            i = int(min(n[b], ref.n[b]))
            gap = abs(float(inp.ua[b, i]) - float(ref.thr[b, i]))
            kind = "accept"
        else:
            u = float(inp.ur[b])
            gap = min(abs(u - ref.draw_lo[b]), abs(u - ref.draw_hi[b]))
            kind = "draw"
        if gap < TOL_U:
            near += 1
        else:
            hard += 1
            detail.append((b, kind, gap))
    return Report(B * (k + 1), B, mism, near, hard, detail[:10])


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
