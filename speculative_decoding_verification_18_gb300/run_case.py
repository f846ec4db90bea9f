"""Run the one-call verify a few times on a named workload (for profilers).

    python -m speculative_decoding_verification_18_gb300.run_case c4 --batch 64 --path 3 --reps 4
    python -m speculative_decoding_verification_18_gb300.run_case c3 --match

Builds the seeded inputs of the workload (optionally with another batch size),
copies them to the GPU, and calls spec_verify_sample / spec_verify_greedy
`reps` times on one stream, then prints the status word.  `--path` forces the
two-kernel (1), fused (2) or row-skipping (3) path; 0 keeps the automatic
choice; `--draw-mode` the sampled draw (1 split, 2 cluster); `--match` runs the sample-and-match verify (spec_verify_match) on a
sampled workload instead.  Nothing is timed here: the point is a fixed, short sequence of
launches that a profiler can select from with its skip / count options.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import inputs as I
from . import specverify as sv


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("workload", choices=sorted(I.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0, help="override B (0: the workload's)")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2, 3])
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--match", action="store_true", help="sample-and-match verify")
    ap.add_argument("--draw-mode", type=int, default=0, choices=[0, 1, 2],
                    help="sampled draw: 1 split, 2 cluster (0 automatic)")
    a = ap.parse_args(argv)
    kw = dict(I.WORKLOADS[a.workload])
    if a.batch > 0:
        kw["B"] = a.batch
    inp = I.make_inputs(**kw)
    dev = torch.device("cuda", 0)
    if inp.dtype == "bf16":
        logits = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        logits = torch.from_numpy(inp.logits).to(dev)
    x = torch.from_numpy(inp.x).to(dev)
    B, k, V = inp.B, inp.k, inp.V
    ws = sv.workspace(B, k, V, logits.dtype, dev)
    out = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    tu = sv.Tuning(path=a.path, draw_mode=a.draw_mode) if (a.path or a.draw_mode) else None
    if inp.mode == "greedy":
        for _ in range(a.reps):
            sv.spec_verify_greedy(logits, x, out, n, ws, tuning=tu)
    elif a.match:
        ua = torch.from_numpy(inp.ua).to(dev)
        ur = torch.from_numpy(inp.ur).to(dev)
        for _ in range(a.reps):
            sv.spec_verify_match(logits, x, ua, ur, inp.T, out, n, ws, tuning=tu)
    else:
        q = torch.from_numpy(inp.q).to(dev)
        ua = torch.from_numpy(inp.ua).to(dev)
        ur = torch.from_numpy(inp.ur).to(dev)
        for _ in range(a.reps):
            sv.spec_verify_sample(logits, q, x, ua, ur, inp.T, out, n, ws, tuning=tu)
    torch.cuda.synchronize(dev)
    st, bits, ndeg = sv.spec_verify_read_status(ws)
    print(f"{a.workload} B={B} k={k} V={V} path={a.path} draw_mode={a.draw_mode} match={a.match} "
          f"reps={a.reps}: status {st} "
          f"bits {bits:#x} degenerate {ndeg}")


if __name__ == "__main__":
    main()
