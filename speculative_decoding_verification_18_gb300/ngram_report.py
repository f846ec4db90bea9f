"""Timing of the n-gram drafter kernel on synthetic repeating token streams.

    python -m speculative_decoding_verification_18_gb300.ngram_report [--B 256] [--L 8192]

Histories of B sequences (up to L tokens, lengths uniform in [L/2, L]) are
rotated over enough device copies to exceed the L2; a CUDA graph of drafter
calls is replayed and timed with CUDA events.  The kernel reads every history
token at least once: the report gives that byte count per call over the time,
and the fraction of the measured copy bandwidth (MEASURED_PEAKS.json when
present).
"""
from __future__ import annotations

import argparse
import json
import os

import torch

from . import inputs as I
from . import specverify as sv

L2_BYTES = 129 * 1024 * 1024


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--B", type=int, default=256)
    ap.add_argument("--L", type=int, default=8192)
    ap.add_argument("--k", type=int, default=8)
    ap.add_argument("--n-min", type=int, default=1)
    ap.add_argument("--n-max", type=int, default=4)
    ap.add_argument("--reps", type=int, default=200)
    a = ap.parse_args(argv)
    hist, lengths = I.ngram_histories(a.B, a.L, seed=11)
    set_bytes = hist.nbytes
    copies = int(min(32, max(1, -(-2 * L2_BYTES // set_bytes))))
    hs = [torch.from_numpy(hist).cuda() for _ in range(copies)]
    ls = [torch.from_numpy(lengths).cuda() for _ in range(copies)]
    ds = [torch.empty((a.B, a.k), dtype=torch.int32, device="cuda") for _ in range(copies)]
    ns = [torch.empty(a.B, dtype=torch.int32, device="cuda") for _ in range(copies)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(copies):
            sv.spec_ngram_draft(hs[i], ls[i], a.k, a.n_min, a.n_max, ds[i], ns[i])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(copies):
                sv.spec_ngram_draft(hs[i], ls[i], a.k, a.n_min, a.n_max, ds[i], ns[i])
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = max(1, a.reps // copies)
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * copies)
    tokens = int(lengths.sum())
    gbs = tokens * 4 / (us * 1e-6) / 1e9
    peak = None
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peak = float(json.load(f)["hbm_gbs"])
    except Exception:
        pass
    drafted = float((ns[0].cpu() > 0).float().mean())
    print(json.dumps({"kernel": "sv_ngram_kernel", "B": a.B, "Lmax": a.L, "k": a.k,
                      "n_min": a.n_min, "n_max": a.n_max, "us_per_call": round(us, 3),
                      "history_tokens": tokens, "gbs": round(gbs, 1),
                      "frac_of_measured_copy": round(gbs / peak, 4) if peak else None,
                      "share_with_draft": round(drafted, 3), "copies": copies}))


if __name__ == "__main__":
    main()
