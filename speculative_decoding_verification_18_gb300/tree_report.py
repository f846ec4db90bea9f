"""Timing of tree verification (spec_verify_tree) on synthetic drafted trees.

    python -m speculative_decoding_verification_18_gb300.tree_report [--mode sample]
        [--B 64] [--N 16] [--V 32000] [--dtype bf16] [--branching 4,2,2]

A batch of B trees of N nodes (the level-by-level shape of ``--branching``,
Zipf logits, drafts drawn from q at each node) is copied to enough device
copies to exceed the L2; CUDA graphs of whole calls, and of the row stream
alone (spec_verify_rows over the same B*N rows), are replayed and timed with
CUDA events.  Prints one JSON line: us per call, tree rows (B*N) per second,
the row stream's time and algorithmic GB/s (B*N*V logits) as a fraction of the
measured copy bandwidth (MEASURED_PEAKS.json when present), the walk's share,
and the mean accepted path length.
"""
from __future__ import annotations

import argparse
import json
import os

import numpy as np
import torch

from . import inputs as I
from . import specverify as sv

L2_BYTES = 129 * 1024 * 1024


def _graph_us(fns, reps):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for f in fns:
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for f in fns:
                f()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(fns))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--mode", default="sample", choices=["sample", "greedy"])
    ap.add_argument("--B", type=int, default=64)
    ap.add_argument("--N", type=int, default=16)
    ap.add_argument("--V", type=int, default=32000)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32"])
    ap.add_argument("--T", type=float, default=1.0)
    ap.add_argument("--branching", default="4,2,2")
    ap.add_argument("--reps", type=int, default=40)
    a = ap.parse_args(argv)
    br = tuple(int(v) for v in a.branching.split(","))
    t = I.make_tree_inputs(mode=a.mode, B=a.B, N=a.N, V=a.V, dtype=a.dtype, T=a.T,
                           branching=br, draft_sigma=0.5, seed=17)
    B, N, V = t.B, t.N, t.V
    set_bytes = t.logits.nbytes + (t.q.nbytes if t.q is not None else 0)
    copies = int(min(16, max(1, -(-2 * L2_BYTES // set_bytes))))
    dev = torch.device("cuda", 0)

    def dev_set():
        if t.dtype == "bf16":
            lg = torch.from_numpy(t.logits.view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            lg = torch.from_numpy(t.logits).to(dev)
        d = dict(lg=lg, tok=torch.from_numpy(t.tok).to(dev), par=torch.from_numpy(t.par).to(dev),
                 x=torch.from_numpy(np.ascontiguousarray(t.tok[:, 1:])).to(dev))
        if t.mode == "sample":
            d.update(q=torch.from_numpy(t.q).to(dev), ua=torch.from_numpy(t.ua).to(dev),
                     ur=torch.from_numpy(t.ur).to(dev))
        return d

    sets = [dev_set() for _ in range(copies)]
    ws = [sv.workspace(B, N - 1, V, sets[0]["lg"].dtype, dev) for _ in range(copies)]
    out = torch.empty((B, N), dtype=torch.int32, device=dev)
    nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    mode = sv.SV_MODE_SAMPLE if t.mode == "sample" else sv.SV_MODE_GREEDY

    def call(i):
        d = sets[i]
        return lambda: sv.spec_verify_tree(mode, d["lg"], d.get("q"), d["tok"], d["par"],
                                           d.get("ua"), d.get("ur"), t.T, out, nodes, n, ws[i])

    def rows(i):
        d = sets[i]
        return lambda: sv.spec_verify_rows(mode, d["lg"], d.get("q"), d["x"], t.T, ws[i])

    reps = max(3, a.reps // copies)
    us_call = _graph_us([call(i) for i in range(copies)], reps)
    us_rows = _graph_us([rows(i) for i in range(copies)], reps)
    call(0)()
    torch.cuda.synchronize()
    mean_n = float(n.float().mean())
    peak = None
    try:
        with open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                               "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["hbm_gbs"])
    except Exception:
        pass
    rows_gbs = t.logits.nbytes / (us_rows * 1e-6) / 1e9
    print(json.dumps({
        "call": "spec_verify_tree", "mode": t.mode, "B": B, "N": N, "V": V, "dtype": t.dtype,
        "branching": list(br), "us_per_call": round(us_call, 2),
        "tree_rows_per_s": round(B * N / (us_call * 1e-6), 1),
        "row_stream_us": round(us_rows, 2), "row_stream_gbs": round(rows_gbs, 1),
        "row_stream_frac_of_measured_copy": round(rows_gbs / peak, 4) if peak else None,
        "walk_us": round(us_call - us_rows, 2), "mean_accepted": round(mean_n, 3),
        "copies": copies}))


if __name__ == "__main__":
    main()
