#!/usr/bin/env python3
"""Benchmark of the batched speculative-decoding verify step on GB300.

One step = one verify of one batch of the named workload (default c4, the
largest: sampled, B=256, k=8, V=151936, fp32 logits, T=1): the row stream, the
accept scan and the draw.  Metric: verify rows per second, rows = B*(k+1) per
step, summed over GPUs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c1..c5]
                  [--impl ours|reference]

Timing: inputs are resident in HBM and rotated over enough copies to exceed the
129 MB L2 between reuses; exactly W warm-up steps, then exactly K timed steps,
replayed from CUDA graphs (one graph of `copies` consecutive verifies, and one
of the first K mod copies for the remainder) and timed with CUDA events on the
launching stream, bracketed by a barrier and a device synchronisation, max over
ranks.
Each kernel of the path the one-call API takes is timed the same way for the
roofline figure (the fused kernel is the whole verify; on the two-stage paths
the row stream and the draw kernel are replayed alone), and the slower one is
reported.  `e2e` repeats the measurement through the same C ABI with
the inputs in pinned HOST memory: every step copies its inputs host-to-device,
verifies and copies the outputs back.  `cpu_baseline` times the float64 oracle
on a bounded sample on this host's cores (and on one core), and its outputs on
the timed inputs are compared with the GPU's (mismatches, near-threshold cases);
the realised acceptance rate alpha = sum min(p, q) of the inputs is reported
beside the measured acceptance.  With --impl reference the oracle is the
reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_18_gb300 import inputs as I  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: about 2 s worth)")
    ap.add_argument("--warmup", type=int, default=10, help="warm-up steps (at least 3)")
    ap.add_argument("--workload", default="c4", choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# Sections of specverify.cu (between its '// ----' headers) that every kernel's
# code draws on, and the kernels that also run the draw.
_COMMON_SECTIONS = ("workspace", "small helpers", "online softmax partials")
_DRAWING = ("sv_verify_kernel", "sv_finish_sample_kernel", "sv_precise_kernel",
            "sv_match_draw_kernel", "sv_split_draw_kernel", "sv_split_precise_kernel")


def kernel_source_hash(kernel=None):
    """Hash of the sources a kernel's counters depend on: the section of
    specverify.cu that defines it, the common device sections, the draw
    section for kernels that draw, and ff.cuh; the whole file when the kernel
    is not found.  A stage of several kernels ('a+b') takes the union of their
    sections."""
    csrc = os.path.join(ROOT, "speculative_decoding_verification_18_gb300", "csrc")
    with open(os.path.join(csrc, "specverify.cu")) as fh:
        text = fh.read()
    if kernel:
        heads = [(h.start(), h.group(1).strip())
                 for h in re.finditer(r"^// -{40,} (.*)$", text, re.M)]
        bounds = [(a, heads[i + 1][0] if i + 1 < len(heads) else len(text), name)
                  for i, (a, name) in enumerate(heads)]
        keep, found = set(), True
        for kn in kernel.split("+"):
            m = re.search(r"__global__[^;{]*?\b" + re.escape(kn) + r"\s*\(", text)
            if not m:
                found = False
                break
            want = set(_COMMON_SECTIONS) | ({"draw phase"} if kn in _DRAWING else set())
            keep |= {i for i, (a, b, name) in enumerate(bounds)
                     if name in want or a <= m.start() < b}
        if found:
            text = "".join(text[bounds[i][0]:bounds[i][1]] for i in sorted(keep))
    h = hashlib.sha256(text.encode())
    with open(os.path.join(csrc, "ff.cuh"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload, kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it was
    captured from the current kernel source; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes_rows(inp):
    """Bytes the row-stream kernel must move per launch: every logits row once, the
    draft tokens, the gathered l(x) / q(x) (one 32-byte sector each), the records."""
    R = inp.B * (inp.k + 1)
    esz = 2 if inp.dtype == "bf16" else 4
    b = R * inp.V * esz + inp.B * inp.k * 4 + R * 32
    b += inp.B * inp.k * 32 * (2 if inp.mode == "sample" else 1)
    return b


def algorithmic_bytes_fused(inp, n):
    """Bytes the fused kernel must move for one verify with the realised accepted
    lengths n: logits rows 0..n_b of every sequence (later rows are never needed),
    the q row of each rejection (the residual), tokens, uniforms, gathers, outputs."""
    esz = 2 if inp.dtype == "bf16" else 4
    n = np.asarray(n, dtype=np.int64)
    rows = int(np.sum(np.clip(n, 0, inp.k) + 1))
    b = rows * inp.V * esz
    if inp.mode == "sample":
        b += int(np.sum(n < inp.k)) * inp.V * 4 + inp.B * inp.k * 4 + inp.B * 4
    b += inp.B * inp.k * 4 + inp.B * inp.k * 32 * (2 if inp.mode == "sample" else 1)
    b += inp.B * (inp.k + 2) * 4
    return b


def algorithmic_bytes_rows_needed(inp, n):
    """Bytes the row stream must move when it reads only the rows the scan needs
    (0..n_b of every sequence), with their gathers, and writes every record."""
    esz = 2 if inp.dtype == "bf16" else 4
    n = np.asarray(n, dtype=np.int64)
    rows = int(np.sum(np.clip(n, 0, inp.k) + 1))
    b = rows * inp.V * esz + inp.B * (inp.k + 1) * 32
    b += inp.B * inp.k * 4 + inp.B * inp.k * 32 * (2 if inp.mode == "sample" else 1)
    if inp.mode == "sample":
        b += inp.B * inp.k * 4
    return b


def algorithmic_bytes_draw(inp, n):
    """Bytes the draw kernel must move: the records of each sequence and, in
    sampled mode, its decision row once and the q row of a rejection, the
    uniforms, the outputs."""
    esz = 2 if inp.dtype == "bf16" else 4
    n = np.asarray(n, dtype=np.int64)
    b = inp.B * (inp.k + 1) * 32 + inp.B * inp.k * 4 + inp.B * (inp.k + 2) * 4
    if inp.mode == "sample":
        b += inp.B * inp.V * esz + int(np.sum(n < inp.k)) * inp.V * 4 + inp.B * (inp.k + 1) * 4
    return b


def full_tensor_bytes(inp):
    """logits + draft_probs + small inputs (the convention of the headline metric)."""
    b = inp.logits.nbytes + inp.x.nbytes
    if inp.mode == "sample":
        b += inp.q.nbytes + inp.ua.nbytes + inp.ur.nbytes
    return b


def oracle_time(inp, seqs, nthreads, min_seconds=3.0, min_reps=2):
    """Seconds per call of the oracle on the first `seqs` sequences."""
    import oracle
    oracle.build()
    sl = slice(0, seqs)
    args = (oracle.GREEDY if inp.mode == "greedy" else oracle.SAMPLE, inp.logits[sl], inp.dtype,
            None if inp.q is None else inp.q[sl], inp.x[sl],
            None if inp.ua is None else inp.ua[sl], None if inp.ur is None else inp.ur[sl],
            inp.T if inp.mode == "sample" else 1.0)
    reps, t0 = 0, time.perf_counter()
    while reps < min_reps or time.perf_counter() - t0 < min_seconds:
        oracle.verify_batch(*args, nthreads=nthreads)
        reps += 1
    return (time.perf_counter() - t0) / reps


def oracle_parity(inp, out, n, nthreads):
    """The oracle on the whole timed batch, compared with the GPU's outputs by
    the parity rule (greedy: equal; sampled: equal up to decisions whose uniform
    lies within 1e-5 of the oracle's threshold)."""
    import oracle
    mode = oracle.GREEDY if inp.mode == "greedy" else oracle.SAMPLE
    ref = oracle.verify_batch(mode, inp.logits, inp.dtype, inp.q, inp.x, inp.ua, inp.ur,
                              inp.T if inp.mode == "sample" else 1.0, nthreads=nthreads)
    c = oracle.compare_outputs(inp.mode, inp.ua, inp.ur, out, n, ref, 1e-5)
    return {"rows": c.rows, "sequences": c.sequences,
            "mismatched_sequences": c.mismatched_sequences,
            "near_threshold": c.near_threshold, "hard": c.hard}


def acceptance_report(inp, n_all):
    """Realised acceptance of the timed inputs: alpha = sum_v min(p_i(v), q_i(v))
    per drafted row (the chance a draft from q is accepted), its mean over the
    batch, and the measured accepted fraction and tokens per verify."""
    n = np.concatenate([np.asarray(v) for v in n_all])
    rep = {"accepted_fraction": float(np.clip(n, 0, None).mean() / inp.k),
           "tokens_per_verify": float((np.clip(n, 0, None) + 1).mean())}
    if inp.mode != "sample":
        return rep
    lv = inp.logits_f32()
    al = []
    for b in range(inp.B):
        z = lv[b, :inp.k].astype(np.float64) / inp.T
        z -= z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        al.append(np.minimum(p, inp.q[b]).sum(axis=1))
    al = np.concatenate(al)
    rep.update(alpha_mean=float(al.mean()), alpha_min=float(al.min()),
               alpha_max=float(al.max()))
    return rep


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of the ranks' values (a job's time is its slowest rank's);
    `dist` is torch.distributed with a process group, or None for one rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units: float, ms: float) -> float:
    """Units processed by all ranks per second of the job's time."""
    return units / (ms / 1e3)


def run_reference(args, world, rank):
    """The reference arm: the float64 oracle on this host's cores, same workload."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = I.workload(args.workload)
    nt = cores()
    steps = args.steps if args.steps > 0 else 5
    per_seq = oracle_time(inp, 1, nt, min_seconds=0.5, min_reps=1)
    budget = 120.0 / max(1, steps + args.warmup)
    seqs = int(max(1, min(inp.B, budget / max(per_seq, 1e-9))))
    sl = slice(0, seqs)
    call = lambda: oracle.verify_batch(
        oracle.GREEDY if inp.mode == "greedy" else oracle.SAMPLE, inp.logits[sl], inp.dtype,
        None if inp.q is None else inp.q[sl], inp.x[sl], None if inp.ua is None else inp.ua[sl],
        None if inp.ur is None else inp.ur[sl], inp.T if inp.mode == "sample" else 1.0,
        nthreads=nt)
    for _ in range(args.warmup):
        call()
    t0 = time.perf_counter()
    for _ in range(steps):
        call()
    dt = time.perf_counter() - t0
    rows = seqs * (inp.k + 1) * steps
    value = rows / dt
    sample = f"first {seqs} of {inp.B} sequences per step ({seqs * (inp.k + 1)} rows)"
    line = {
        "impl": "reference", "metric": "verify rows/s", "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {I.WORKLOAD_NAMES[args.workload]}",
                   "B": inp.B, "k": inp.k, "V": inp.V, "logits_dtype": inp.dtype,
                   "mode": inp.mode},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nt, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        if world > 1:
            # Rank 0 alone runs the CPU reference; the others exit without work.
            run_reference(args, world, rank)
            return
        run_reference(args, world, rank)
        return

    import torch
    from speculative_decoding_verification_18_gb300 import build as libbuild
    from speculative_decoding_verification_18_gb300 import specverify as sv

    libbuild.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    inp = I.workload(args.workload)
    B, k, V = inp.B, inp.k, inp.V
    rows_per_step = B * (k + 1)
    set_bytes = inp.logits.nbytes + (0 if inp.q is None else inp.q.nbytes)
    copies = int(min(16, max(1, -(-2 * L2_BYTES // set_bytes))))

    # Device-resident inputs, rotated over `copies` distinct buffers.
    def dev_set():
        if inp.dtype == "bf16":
            lg = torch.from_numpy(inp.logits.view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            lg = torch.from_numpy(inp.logits).to(dev)
        d = {"logits": lg, "x": torch.from_numpy(inp.x).to(dev)}
        if inp.mode == "sample":
            d["q"] = torch.from_numpy(inp.q).to(dev)
            d["ua"] = torch.from_numpy(inp.ua).to(dev)
            d["ur"] = torch.from_numpy(inp.ur).to(dev)
        return d

    sets = [dev_set() for _ in range(copies)]
    path = sv.debug_path(sv.SV_MODE_GREEDY if inp.mode == "greedy" else sv.SV_MODE_SAMPLE, B, V,
                         inp.dtype)
    fused = path == sv.PATH_FUSED
    # greedy batches of about one row per resident CTA take the flat row stream
    flat_ctas = sv.debug_flat_ctas(B, k, V, inp.dtype) if inp.mode == "greedy" else 0
    rows_kname = "sv_flat_greedy_kernel" if flat_ctas else "sv_rows_kernel"
    ws = [sv.workspace(B, k, V, sets[0]["logits"].dtype, dev) for _ in range(copies)]
    outs = [torch.empty((B, k + 1), dtype=torch.int32, device=dev) for _ in range(copies)]
    ns = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(copies)]

    def verify(i, stream=None):
        s = sets[i]
        if inp.mode == "greedy":
            sv.spec_verify_greedy(s["logits"], s["x"], outs[i], ns[i], ws[i], stream)
        else:
            sv.spec_verify_sample(s["logits"], s["q"], s["x"], s["ua"], s["ur"], inp.T, outs[i],
                                  ns[i], ws[i], stream)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(copies):
            verify(i)  # device set-up outside capture
    torch.cuda.synchronize(dev)
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    verify(i)
        torch.cuda.synchronize(dev)
        return g

    graph = capture(copies)
    partial = {}

    def run_steps(n):
        """Exactly n verify steps: whole graphs of `copies` steps, then a graph of
        the first n mod copies."""
        for _ in range(n // copies):
            graph.replay()
        r = n % copies
        if r:
            if r not in partial:
                partial[r] = capture(r)
            partial[r].replay()

    # Exactly W warm-up steps (at least 3), then K (if not given, about 2 s of steps).
    W = max(3, args.warmup)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        run_steps(W)
    torch.cuda.synchronize(dev)
    est = (time.perf_counter() - t0) / W
    K = args.steps if args.steps > 0 else int(min(200000, max(copies, 2.0 / max(est, 1e-7))))
    if K % copies and (K % copies) not in partial:
        partial[K % copies] = capture(K % copies)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    except Exception:
        pass

    # ---- timed region
    # nvidia-smi samples every 200 ms, far longer than a short timed region: the
    # same steps run untimed for half a second on each side of it (whole graphs
    # in batches of about 50 ms), so that the samples around the K timed steps
    # see this load.
    n_load = copies * max(1, int(0.05 / max(est, 1e-7)) // copies)

    def load_for(seconds):
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            with torch.cuda.stream(stream):
                run_steps(n_load)
            torch.cuda.synchronize(dev)

    sampler = ClockSampler(uuid)
    with sampler:
        load_for(0.5)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            run_steps(K)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        ms = ev0.elapsed_time(ev1)
        load_for(0.5)

        # Each kernel of the one-call path timed alone: the fused kernel is the
        # whole verify (the loop above); the two-stage paths' row stream and draw
        # kernel are replayed from graphs of their own over the same rotated inputs
        # (the draw graph reads the row records the row-stream graph left).
        mode = sv.SV_MODE_GREEDY if inp.mode == "greedy" else sv.SV_MODE_SAMPLE

        def stage_ms(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    for i in range(copies):
                        fn(i)
                g.replay()
                torch.cuda.synchronize(dev)
                r1 = max(1, -(-K // copies) // 2)
                a0 = torch.cuda.Event(enable_timing=True)
                a1 = torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for _ in range(r1):
                    g.replay()
                a1.record(stream)
            torch.cuda.synchronize(dev)
            return a0.elapsed_time(a1) / (r1 * copies)

        def rows_stage(i):
            s = sets[i]
            if path == sv.PATH_SKIP:
                sv.debug_rows_skip(mode, s["logits"], s.get("q"), s["x"], s.get("ua"), inp.T,
                                   ws[i])
            else:
                sv.spec_verify_rows(mode, s["logits"], s.get("q"), s["x"], inp.T, ws[i])

        def finish_stage(i):
            s = sets[i]
            sv.spec_verify_finish(mode, s["logits"], s.get("q"), s["x"], s.get("ua"), s.get("ur"),
                                  inp.T, outs[i], ns[i], ws[i])

        if fused:
            stage_times = {"sv_verify_kernel": ms / K}
        else:
            # the draw stage of a large sampled batch is two kernels: the fast draw
            # and the precise draws it hands on
            fin_name = ("sv_finish_greedy_kernel" if inp.mode == "greedy"
                        else "sv_split_draw_kernel+sv_split_precise_kernel")
            stage_times = {rows_kname: stage_ms(rows_stage),
                           fin_name: stage_ms(finish_stage)}
    clocks = sampler.summary()
    clocks["window"] = (f"the {K} timed steps with 0.5 s of the same steps untimed before and "
                        f"after them, then the per-stage replays")

    ms = max_over_ranks(ms, dist, dev)
    value = job_rate(rows_per_step * K * world, ms)

    # ---- end to end through the C ABI with host buffers
    pin = lambda a: torch.from_numpy(a).pin_memory()
    h_logits = pin(inp.logits.view(np.int16) if inp.dtype == "bf16" else inp.logits)
    h = {"logits": h_logits, "x": pin(inp.x)}
    if inp.mode == "sample":
        h.update(q=pin(inp.q), ua=pin(inp.ua), ur=pin(inp.ur))
    h_out = torch.empty((B, k + 1), dtype=torch.int32).pin_memory()
    h_n = torch.empty(B, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = h_out.numel() * 4 + h_n.numel() * 4
    e2e_steps = int(max(3, min(K, 2.0 / max(est * 4 + h2d / 200e9, 1e-7))))

    def e2e_step():
        s = sets[0]
        if inp.dtype == "bf16":
            s["logits"].view(torch.int16).copy_(h["logits"], non_blocking=True)
        else:
            s["logits"].copy_(h["logits"], non_blocking=True)
        for key in h:
            if key != "logits":
                s[key].copy_(h[key], non_blocking=True)
        verify(0)
        h_out.copy_(outs[0], non_blocking=True)
        h_n.copy_(ns[0], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = job_rate(rows_per_step * e2e_steps * world, e2e_ms)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel
    peak, peak_src = measured_peaks()
    n_all = [nn.cpu().numpy() for nn in ns]
    rows_read = None
    if path == sv.PATH_SKIP:  # rows the position-major stream actually read (copy 0)
        st0 = sv.spec_verify_row_stats(ws[0], B, k)
        rows_read = int((st0["argmax"] >= 0).sum())

    def alg_bytes(kname):
        if kname == "sv_verify_kernel":
            return int(np.mean([algorithmic_bytes_fused(inp, nn) for nn in n_all]))
        if kname in ("sv_rows_kernel", "sv_flat_greedy_kernel"):
            if path == sv.PATH_SKIP:
                return int(np.mean([algorithmic_bytes_rows_needed(inp, nn) for nn in n_all]))
            return algorithmic_bytes_rows(inp)
        return int(np.mean([algorithmic_bytes_draw(inp, nn) for nn in n_all]))

    stages = {}
    for kname, kms in stage_times.items():
        alg = alg_bytes(kname)
        stages[kname] = {"ms": round(kms, 5), "algorithmic_bytes": alg,
                         "achieved_gbs": round(alg / (kms / 1e3) / 1e9, 1)}
    kname = max(stage_times, key=stage_times.get)
    k1_ms = stage_times[kname]
    alg = stages[kname]["algorithmic_bytes"]
    achieved = alg / (k1_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic(args.workload, kname),
                "kernel": kname, "kernel_ms": round(k1_ms, 5),
                "algorithmic_bytes": alg, "peak_source": peak_src + " (copy bandwidth)",
                "stages": stages,
                "full_tensor_gbs": round(full_tensor_bytes(inp) / (ms / K / 1e3) / 1e9, 1)}
    # The whole step against the HBM floor: the algorithmic bytes of every stage
    # at the measured copy bandwidth, over the measured time per step.
    step_bytes = sum(v["algorithmic_bytes"] for v in stages.values())
    roofline["step_algorithmic_bytes"] = step_bytes
    roofline["hbm_floor_frac"] = round((step_bytes / (peak * 1e9)) / (ms / K / 1e3), 4)
    if rows_read is not None:
        roofline["rows_read"] = rows_read
        roofline["rows_needed"] = int(np.mean([np.sum(np.clip(nn, 0, k) + 1) for nn in n_all]))

    # ---- CPU baseline: the oracle on a bounded sample, on every core and on one
    nt = cores()
    per_call = oracle_time(inp, min(B, 1), nt, min_seconds=0.2, min_reps=1)
    seqs = int(max(1, min(B, 5.0 / max(per_call, 1e-9))))
    t_cpu = oracle_time(inp, seqs, nt, min_seconds=5.0, min_reps=2)
    cpu_value = seqs * (k + 1) / t_cpu
    seqs1 = int(max(1, min(B, 3.0 / max(per_call * nt, 1e-9))))
    t_cpu1 = oracle_time(inp, seqs1, 1, min_seconds=3.0, min_reps=1)
    cpu_value1 = seqs1 * (k + 1) / t_cpu1

    # ---- the oracle on the whole timed batch against the GPU's outputs (copy 0)
    parity = oracle_parity(inp, outs[0].cpu().numpy(), ns[0].cpu().numpy(), nt)
    if inp.mode == "sample":  # draws of copy 0 that needed the float-float pass
        parity["precise_draws"] = sv.debug_status_counts(ws[0])[5]
    accept = acceptance_report(inp, n_all)

    line = {
        "metric": "verify rows/s", "value": value, "unit": "rows/s", "n_gpus": world,
        "sequences_per_s": value / (k + 1),
        "steps": K, "warmup": W, "ms_per_step": ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {I.WORKLOAD_NAMES[args.workload]}",
                   "B": B, "k": k, "V": V, "logits_dtype": inp.dtype, "mode": inp.mode,
                   "T": inp.T, "rows_per_step": rows_per_step,
                   "l2": f"inputs rotated over {copies} device copies "
                         f"({copies * set_bytes / 2**20:.0f} MiB > 129 MB L2)",
                   "timing": f"{K // copies} replays of a CUDA graph of {copies} verifies"
                             + (f" and one of {K % copies}" if K % copies else ""),
                   "path": {sv.PATH_FUSED: "fused per-sequence kernel",
                            sv.PATH_SKIP: "position-major row stream with row skipping + "
                                          + ("finish kernel" if inp.mode == "greedy"
                                             else "split draw + split precise pass"),
                            sv.PATH_TWO_KERNEL: "row stream + "
                                                + ("finish kernel" if inp.mode == "greedy"
                                                   else "split draw + split precise pass")}[path]
                           + (f" (flat greedy stream over {flat_ctas} CTAs)" if flat_ctas else ""),
                   "parallelism": f"replicas x{world}"},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": (1 if fused else 3 if inp.mode == "sample" else 2) * K,
        "roofline": roofline,
        "cpu_baseline": {"value": cpu_value, "unit": "rows/s", "cores": nt, "kind": "oracle",
                         "sample": f"first {seqs} of {B} sequences ({seqs * (k + 1)} rows), "
                                   f"repeated for >= 5 s",
                         "value_1_thread": cpu_value1,
                         "sample_1_thread": f"first {seqs1} of {B} sequences, one thread, "
                                            f"repeated for >= 3 s"},
        "parity": parity,
        "acceptance": accept,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
